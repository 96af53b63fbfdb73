// Compression stage of 1-bit LAMB (arXiv 2104.06069): the fused worker +
// server pass (templates; instantiated by k_compress_*.cu).
//
// One CTA owns a tile of whole chunks for all W virtual workers, so the
// "communication" of the compressed allreduce (section 5 summary: gather chunk
// k of every worker at server k, average, scatter the average) happens in
// registers: the worker loop accumulates each element's server sum while the
// worker's sign bits are still live, and the packed words and scales are also
// written to the exchange buffers (signs_w, scale_w) as the message.
//
// Data movement: CTAs are persistent (tile t = blockIdx.x + i*gridDim.x; a
// tile is 4096 elements = 4096/C chunks, or one 8192-element chunk).
// Every input of a tile -- the old momentum (after the first compression
// step: the last server message, sign words and chunk scales, 1/32 of the
// bytes; m is exactly sign x scale, so no dense copy is kept), each worker's
// gradient and error, then the server error, the frozen preconditioner
// sqrt(v) + eps and the fresh second moment -- is copied into a 7-slot ring of shared-memory slots by TMA bulk
// copies (cp.async.bulk, completion on one mbarrier per slot), issued by
// thread 0 as soon as enough slots are released, so the next arrays stream
// in while the CTA reduces and stores the current one; while the server phase
// holds its three arrays the next tile's momentum and first worker are
// already loading.  Outputs are written with coalesced 16-byte stores.
//
// Thread map: thread `tid` of an NT-thread CTA holds SLOTS aligned float4
// groups, group s at chunk offset s*NT*4 + tid*4.  Warp w's lanes therefore
// cover the 128 consecutive elements starting at s*NT*4 + w*128, which is one
// leaf block of the canonical pairwise tree.
#pragma once
#include <atomic>
#include <type_traits>

#include "lamb1b_internal.cuh"

namespace lamb1b {

// ---- TMA bulk copies and mbarriers (inline PTX, sm_90+) ----------------------
namespace tma {

__device__ __forceinline__ uint32_t saddr(const void* p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void bar_init(uint64_t* bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(saddr(bar)), "r"(count) : "memory");
}

// makes the initialised barriers visible to the asynchronous (TMA) proxy
__device__ __forceinline__ void fence_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;\n\tfence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void arrive_expect_tx(uint64_t* bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(saddr(bar)), "r"(bytes)
                 : "memory");
}

// global -> shared, `bytes` a multiple of 16, both addresses 16-byte aligned
__device__ __forceinline__ void load(void* dst, const void* src, uint32_t bytes, uint64_t* bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(saddr(dst)), "l"(src), "r"(bytes), "r"(saddr(bar))
        : "memory");
}

__device__ __forceinline__ bool try_wait(uint64_t* bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(saddr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

}  // namespace tma

// Bounded wait for a stage: try_wait suspends for a hardware-defined time per
// call, so with the default limit (P.wait_tries = 2^24) this gives up after
// seconds, never hangs.
__device__ __forceinline__ bool wait_stage(uint64_t* bar, uint32_t parity, uint32_t tries)
{
    for (uint32_t it = 0; it < tries; ++it)
        if (tma::try_wait(bar, parity)) return true;
    return false;
}

// Sign words of S slots at once (S a power of two, S <= 8).  In slot s the
// word r of a warp's 128-element block is made of the nibbles nib[s] (4
// consecutive sign bits) of lanes 8r..8r+7.  They are OR-combined across the
// 8 lanes; while a lane still holds n > 1 slots it passes half of them to its
// partner and keeps the other half.  Lane l returns word l/8 of slot
// tree_block<S>(l) (lanes with l % 8 >= S hold duplicates).
template <int S>
__device__ __forceinline__ uint32_t pack_words(const uint32_t (&nib)[S], int lane)
{
    static_assert(S >= 1 && S <= 8 && (S & (S - 1)) == 0, "S a power of two");
    uint32_t v[S];
#pragma unroll
    for (int s = 0; s < S; ++s) v[s] = nib[s] << (4 * (lane & 7));
    int o = 1;
#pragma unroll
    for (int n = S; n > 1; n >>= 1, o <<= 1) {
        const bool hi = (lane & o) != 0;
#pragma unroll
        for (int j = 0; j < n / 2; ++j) {
            const uint32_t send = hi ? v[j] : v[j + n / 2];
            const uint32_t keep = hi ? v[j + n / 2] : v[j];
            v[j] = keep | __shfl_xor_sync(0xFFFFFFFFu, send, o);
        }
    }
    uint32_t t = v[0];
#pragma unroll
    for (; o < 8; o <<= 1) t |= __shfl_xor_sync(0xFFFFFFFFu, t, o);
    return t;
}

template <int GK>
struct GradBytes { static constexpr int value = GK == kGradF32 ? 4 : (GK == kGradBF16 ? 2 : 0); };

// Ring of NSLOT shared-memory slots of TILE floats, one mbarrier per slot.
// Every tile streams, in slot positions: M (m_old, dense or as the last
// server message), then per worker W_w its gradients (when stored) and its
// error, then S (e_s, and for 1-bit LAMB the frozen sqrt(v) + eps), then F
// (v_fresh, 1-bit LAMB only).  Slot position p lives in slot p % NSLOT
// and completes phase (p / NSLOT) of that slot's barrier.  Positions are
// released in order, at the barrier after their last read: a worker's at
// its chunk-norm barrier, S's at the server's, and with late server reads
// (LATE) the frozen preconditioner's and F's at the end of the tile.
template <int TILE>
struct Ring {
    static constexpr uint32_t kSlot = TILE * 4;
};

template <int SG, bool ADAM>
struct Stream {
    static constexpr int kPerWorker = SG > 0 ? 2 : 1;
    static constexpr int kServer = ADAM ? 1 : 2;         // slots of item S
    __device__ static int items(int W) { return W + (ADAM ? 2 : 3); }
    // slots of item r
    __device__ static int slots(int r, int W) { return r == 0 ? 1 : (r <= W ? kPerWorker : (r == W + 1 ? kServer : 1)); }
};

// A slot position kept as (slot, barrier phase), advanced without division.
template <int NSLOT>
struct RingPos {
    int slot = 0;
    uint32_t phase = 0;
    __device__ __forceinline__ RingPos plus(int n) const
    {
        RingPos q = *this;
        q.slot += n;
        if (q.slot >= NSLOT) { q.slot -= NSLOT; q.phase ^= 1u; }
        return q;
    }
};

// Producer side: issue the bulk copies of item r of tile t whose first slot
// position is p (number pos in this CTA's sequence); called by thread 0 only.
// The fault-injection hook leaves out the copy at position P.skip_copy of the
// first CTA, so that the wait for it can only run out.
template <int TILE, int SG, int NSLOT, bool ADAM, bool EB>
__device__ __forceinline__ void issue_item(int64_t t, int r, RingPos<NSLOT> p, int pos,
                                           const Problem& P, const Dev& D, const Grads& G,
                                           unsigned char* ring, uint64_t* full)
{
    using R = Ring<TILE>;
    const int W = P.W;
    const int64_t base = t * TILE;
    constexpr uint32_t kErrBytes = TILE * (EB ? 2 : 4);   // one tile of an error buffer
    const unsigned char* ew = reinterpret_cast<const unsigned char*>(D.e_w);
    const unsigned char* es = reinterpret_cast<const unsigned char*>(D.e_s);
    const int64_t esz = EB ? 2 : 4;
    auto copy = [&](int k, const void* src, uint32_t bytes) {
        if (pos + k == P.skip_copy && blockIdx.x == 0) return;
        const int sl = p.plus(k).slot;
        tma::arrive_expect_tx(&full[sl], bytes);
        tma::load(ring + (uint32_t)sl * R::kSlot, src, bytes, &full[sl]);
    };
    if (r == 0) {
        if (P.m_packed) {
            // the tile's server sign words, then the 16-byte-aligned span of
            // chunk scales that holds its chunks (scale_s is padded by 16)
            if (pos == P.skip_copy && blockIdx.x == 0) return;
            const int64_t k0 = base >> P.log2c;
            const int64_t ka = k0 & ~int64_t(3);
            const uint32_t nsc = (uint32_t)(k0 - ka) + (uint32_t)(TILE >> P.log2c);
            const uint32_t sbytes = (nsc * 4u + 15u) / 16u * 16u;
            const int sl = p.slot;
            tma::arrive_expect_tx(&full[sl], TILE / 8 + sbytes);
            tma::load(ring + (uint32_t)sl * R::kSlot, D.signs_s + base / 32, TILE / 8, &full[sl]);
            tma::load(ring + (uint32_t)sl * R::kSlot + TILE / 8, D.scale_s + ka, sbytes, &full[sl]);
        } else {
            copy(0, D.m + base, R::kSlot);
        }
    } else if (r <= W) {
        const int w = r - 1;
        if constexpr (SG > 0) {
            const int64_t n_t = (base + TILE <= P.N) ? (int64_t)TILE : P.N - base;
            const uint32_t gbytes = (uint32_t)(((n_t * SG) + 15) / 16 * 16);
            copy(0, static_cast<const unsigned char*>(G.ptr) + ((int64_t)w * G.ld + base) * SG, gbytes);
            copy(1, ew + ((int64_t)w * P.Np + base) * esz, kErrBytes);
        } else {
            copy(0, ew + ((int64_t)w * P.Np + base) * esz, kErrBytes);
        }
    } else if (r == W + 1) {
        copy(0, es + base * esz, kErrBytes);
        if constexpr (!ADAM) copy(1, D.d_frz + base, R::kSlot);
    } else {
        copy(0, D.v_fresh + base, R::kSlot);
    }
}

// Plain arrival on an mbarrier (release: this thread's earlier shared-memory
// reads and writes are ordered before it).
__device__ __forceinline__ void bar_arrive(uint64_t* bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(tma::saddr(bar)) : "memory");
}

// One arrival per warp: the warp's lanes synchronise (which orders their
// earlier shared-memory accesses before lane 0's), then lane 0 arrives.
__device__ __forceinline__ void warp_arrive(uint64_t* bar)
{
    __syncwarp();
    if ((threadIdx.x & 31) == 0) bar_arrive(bar);
}

// Wait for phase `parity` of a barrier that other warps of this CTA complete
// (the gradient handoff): bounded like the copy waits (kDefaultWaitTries
// try_wait calls, seconds), and left early once *stop is set (checked every
// 256 tries).  Returns whether the phase completed.
__device__ __forceinline__ bool wait_handoff(uint64_t* bar, uint32_t parity, volatile int* stop)
{
    for (uint32_t it = 0; it < kDefaultWaitTries; ++it) {
        if (tma::try_wait(bar, parity)) return true;
        if ((it & 255u) == 255u && stop && *stop) return false;
    }
    return false;
}

// The same wait for a whole warp (the draw warps, all 32 lanes active):
// every decision is a warp vote, so the lanes always leave together -- none
// can go on to the warp's __syncwarp while another has returned.
__device__ __forceinline__ bool wait_handoff_warp(uint64_t* bar, uint32_t parity, volatile int* stop)
{
    for (uint32_t it = 0; it < kDefaultWaitTries; ++it) {
        if (__all_sync(0xFFFFFFFFu, tma::try_wait(bar, parity))) return true;
        if ((it & 255u) == 255u && __any_sync(0xFFFFFFFFu, *stop != 0)) return false;
    }
    return false;
}

// CTA barriers of the compressing threads.  With draw warps (DRAW) those are
// the first NT threads only, synchronised on named barrier 1; otherwise the
// whole CTA on barrier 0.
template <int NT, bool DRAW>
__device__ __forceinline__ bool sync_or(bool pred)
{
    if constexpr (!DRAW) {
        return __syncthreads_or(pred) != 0;
    } else {
        uint32_t r;
        asm volatile(
            "{\n\t.reg .pred p, q;\n\t"
            "setp.ne.u32 p, %1, 0;\n\t"
            "bar.red.or.pred q, 1, %2, p;\n\t"
            "selp.u32 %0, 1, 0, q;\n\t}"
            : "=r"(r)
            : "r"((uint32_t)pred), "n"(NT)
            : "memory");
        return r != 0;
    }
}

template <int NT, bool DRAW>
__device__ __forceinline__ void sync_all()
{
    if constexpr (!DRAW) __syncthreads();
    else asm volatile("bar.sync 1, %0;" ::"n"(NT) : "memory");
}

// Consumer side: wait for n consecutive slots starting at p.
template <int NSLOT>
__device__ __forceinline__ bool wait_slots(uint64_t* full, RingPos<NSLOT> p, int n, uint32_t tries)
{
    bool ok = true;
    for (int k = 0; k < n; ++k) {
        const RingPos<NSLOT> q = p.plus(k);
        ok &= wait_stage(&full[q.slot], q.phase, tries);
    }
    return ok;
}

// Chunk scale sqrt(S / n).  For a full chunk n = C = 2^log2c, and S / C is
// one multiplication by 2^-log2c (both round the same real number).  The
// square root of a finite value >= 2^-102 uses the generator's sqrt_big, which
// gives the IEEE result on that whole range (lamb1b_gen_selfcheck enumerates
// it); smaller values, zero, infinity, NaN and tail chunks take the rounded
// intrinsics.
template <int C, bool FAST>
__device__ __forceinline__ float chunk_scale(float S, float n)
{
    if (FAST && n == (float)C) {
        constexpr float kInvC = 1.0f / (float)C;       // exact: C is a power of two
        const float m = fmul(S, kInvC);
        return (m >= 0x1p-102f && m <= 0x1.fffffep+127f) ? gen::sqrt_big(m) : fsqrt(m);
    }
    return n > 0.0f ? fsqrt(fdiv(S, n)) : 0.0f;
}

// Chunk totals from the tile's 128-leaf partials red[0 .. NPART) (element
// order).  Each lane loads G = min(4, PPC) consecutive partials with one
// vector load and adds them as the canonical tree does (the level-2 subtrees
// of a chunk's tree); the remaining log2(LPC) butterfly stages, LPC = PPC / G
// lanes per chunk, finish each chunk's tree.  Lanes past LUSED = NPART / G
// repeat lanes lane % LUSED, so every lane returns the total of chunk
// (lane % LUSED) / LPC of the tile.
template <int NPART, int PPC>
struct ChunkLanes {
    static constexpr int G = PPC >= 4 ? 4 : PPC;     // partials per lane
    static constexpr int LPC = PPC / G;              // lanes per chunk
    static constexpr int LUSED = NPART / G;          // lanes with distinct partials
    static_assert(PPC % G == 0 && LUSED >= 1 && LUSED <= 32, "chunk / tile shape");
};

template <int NPART, int PPC>
__device__ __forceinline__ float chunk_totals(const float* red, int lane)
{
    using CL = ChunkLanes<NPART, PPC>;
    const float* r = red + (lane % CL::LUSED) * CL::G;
    float v;
    if constexpr (CL::G == 4) {
        const float4 q = *reinterpret_cast<const float4*>(r);
        v = fadd(fadd(q.x, q.y), fadd(q.z, q.w));
    } else if constexpr (CL::G == 2) {
        const float2 q = *reinterpret_cast<const float2*>(r);
        v = fadd(q.x, q.y);
    } else {
        v = r[0];
    }
#pragma unroll
    for (int o = 1; o < CL::LPC; o <<= 1) v = fadd(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    return v;
}

// A worker's 4 gradients at tile offset off: from its ring slot a (binary32
// or bfloat16 bits, widened exactly), or the values drawn in-kernel (gin).
template <int GK>
__device__ __forceinline__ void load_grad4(const unsigned char* a, int off, const float (&gin)[4],
                                           float g[4])
{
    if constexpr (GK == kGradF32) {
        const float4 v = *reinterpret_cast<const float4*>(a + off * 4);
        g[0] = v.x; g[1] = v.y; g[2] = v.z; g[3] = v.w;
    } else if constexpr (GK == kGradBF16) {
        const uint2 v = *reinterpret_cast<const uint2*>(a + off * 2);
        g[0] = __uint_as_float(v.x << 16);
        g[1] = __uint_as_float(v.x & 0xFFFF0000u);
        g[2] = __uint_as_float(v.y << 16);
        g[3] = __uint_as_float(v.y & 0xFFFF0000u);
    } else {
#pragma unroll
        for (int c = 0; c < 4; ++c) g[c] = gin[c];
    }
}

// Error-buffer element access: 4 consecutive values at element offset off,
// binary32 or (EB) bfloat16 bits widened exactly / rounded to nearest even.
template <bool EB>
__device__ __forceinline__ void load_err4(const void* base, int64_t off, float e[4])
{
    if constexpr (EB) {
        const uint2 v = *reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(base) + off);
        e[0] = __uint_as_float(v.x << 16);
        e[1] = __uint_as_float(v.x & 0xFFFF0000u);
        e[2] = __uint_as_float(v.y << 16);
        e[3] = __uint_as_float(v.y & 0xFFFF0000u);
    } else {
        const float4 v = *reinterpret_cast<const float4*>(static_cast<const float*>(base) + off);
        e[0] = v.x; e[1] = v.y; e[2] = v.z; e[3] = v.w;
    }
}

template <bool EB>
__device__ __forceinline__ void store_err4(void* base, int64_t off, const float e[4])
{
    if constexpr (EB) {
        const uint2 v = make_uint2(bf16x2_bits(e[0], e[1]), bf16x2_bits(e[2], e[3]));
        *reinterpret_cast<uint2*>(static_cast<uint16_t*>(base) + off) = v;
    } else {
        *reinterpret_cast<float4*>(static_cast<float*>(base) + off) = make_float4(e[0], e[1], e[2], e[3]);
    }
}

// CTAs per SM by the size of the copy ring: three when three rings fit in
// shared memory, two for two, else one; a CTA with draw warps (NDRAW > 0)
// runs alone on its SM.
template <int NT, int SLOTS, int NSLOT, int NDRAW = 0>
struct MinBlocks {
    static constexpr int kRing = NSLOT * (NT * 4 * SLOTS) * 4;
    static constexpr int value =
        NDRAW > 0 ? 1 : (kRing <= 72 * 1024 ? 3 : (kRing <= 112 * 1024 ? 2 : 1));
};

// Gradient tiles in flight between the draw warps and the compressing warps.
constexpr int kDrawSlots = 3;

// In-kernel gradients drawn by NDRAW dedicated threads (threads NT ..
// NT+NDRAW-1 of the CTA): for every tile of the CTA and every worker, in the
// order the compressing threads consume them, the tile's TILE gradient
// values (layer_std[l] x N(0,1), or heavy_scale x Student-t(3) in flagged
// tensors; 0 past N) are written into one of kDrawSlots shared-memory slots.
// Slot k is handed over through mbarriers: gfull[k] completes when every
// draw warp has written its part, gempty[k] when every compressing warp has
// read its part (one arrival per warp).  Thread d draws the aligned groups of four at tile offsets
// g*NDRAW*4 + d*4, so one warp writes 512 contiguous bytes per group.  The
// draws are those of the stored-gradient definition (include/lamb1b_gen.h),
// so the values are the same bits wherever they are computed.
template <int TILE, int NDRAW>
__device__ __forceinline__ void draw_gradients(const Problem& P, const Dev& D, const Grads& G,
                                               float* gring, uint64_t* gfull, uint64_t* gempty,
                                               int64_t nloc, volatile int* stop)
{
    constexpr int PG = TILE / (4 * NDRAW);          // groups of four per thread
    static_assert(PG >= 1 && TILE % (4 * NDRAW) == 0, "draw split");
    const int d = threadIdx.x - (int)(blockDim.x - NDRAW);
    RingPos<kDrawSlots> gp;
    for (int64_t ti = 0; ti < nloc; ++ti) {
        const int64_t base = (blockIdx.x + ti * gridDim.x) * (int64_t)TILE;
        float stdv[PG][4];
        uint32_t heavy[PG];
        int nvd[PG];
        {
            int l = D.chunk_l0[base >> P.log2c];
            int64_t lend = D.layer_end[l];
#pragma unroll
            for (int g = 0; g < PG; ++g) {
                const int64_t e = base + g * NDRAW * 4 + d * 4;
                const int64_t r = P.N - e;
                nvd[g] = r >= 4 ? 4 : (r > 0 ? (int)r : 0);
                heavy[g] = 0u;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    stdv[g][c] = 0.0f;
                    if (c < nvd[g]) {
                        while (e + c >= lend) { ++l; lend = D.layer_end[l]; }
                        stdv[g][c] = G.layer_std[l];
                        if (G.layer_heavy && G.layer_heavy[l]) heavy[g] |= 1u << c;
                    }
                }
            }
        }
        bool all_normal = true, all_heavy = true;
#pragma unroll
        for (int g = 0; g < PG; ++g) {
            all_normal = all_normal && heavy[g] == 0u;
            all_heavy = all_heavy && heavy[g] == 0xFu;
        }
        for (int w = 0; w < P.W; ++w) {
            // wait until the compressing threads have read this slot's last
            // tile (a fresh slot passes at once); leave if they stopped
            if (!wait_handoff_warp(&gempty[gp.slot], gp.phase ^ 1u, stop)) {
                if (!*stop) atomicOr(D.flags, 2u);
                return;
            }
            float* slot = gring + gp.slot * TILE;
            // each group of four is stored as soon as it is drawn (past N:
            // zeros; the compressing threads mask those elements)
            auto put = [&](int g, const float (&v)[4]) {
                const float4 q = nvd[g] == 4 ? make_float4(v[0], v[1], v[2], v[3])
                                             : make_float4(nvd[g] > 0 ? v[0] : 0.0f, nvd[g] > 1 ? v[1] : 0.0f,
                                                           nvd[g] > 2 ? v[2] : 0.0f, 0.0f);
                *reinterpret_cast<float4*>(slot + g * NDRAW * 4 + d * 4) = q;
            };
            if (all_heavy) {
                // four independent Student-t chains at a time
#pragma unroll 1
                for (int g = 0; g < PG; ++g) {
                    float v[4];
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        v[c] = fmul(G.heavy_scale,
                                    gen::student_t3(G.seed, base + g * NDRAW * 4 + d * 4 + c, G.t, (uint32_t)w));
                    put(g, v);
                }
            } else {
#pragma unroll
                for (int g = 0; g < PG; ++g) {
                    float v[4];
                    gen::grads_normal4(G.seed, (uint64_t)(base + g * NDRAW * 4 + d * 4) >> 2, G.t,
                                       (uint32_t)w, v);
#pragma unroll
                    for (int c = 0; c < 4; ++c) v[c] = fmul(stdv[g][c], v[c]);
                    if (!all_normal && heavy[g]) {
#pragma unroll
                        for (int c = 0; c < 4; ++c)
                            if ((heavy[g] >> c) & 1u)
                                v[c] = fmul(G.heavy_scale,
                                            gen::student_t3(G.seed, base + g * NDRAW * 4 + d * 4 + c, G.t,
                                                            (uint32_t)w));
                    }
                    put(g, v);
                }
            }
            warp_arrive(&gfull[gp.slot]);
            gp = gp.plus(1);
        }
    }
}

template <int NT, int SLOTS, int GK, int NSLOT, int C, bool ADAM, bool EB, int NDRAW = 0>
__global__ void __launch_bounds__(NT + NDRAW, (MinBlocks<NT, SLOTS, NSLOT, NDRAW>::value))
    k_compress(const Problem P, const Dev D, const Grads G)
{
    constexpr int NWARP = NT / 32;
    constexpr int TILE = NT * 4 * SLOTS;
    constexpr int NPART = TILE / 128;           // 128-leaf partials per tile
    constexpr int PPC = C / 128;                // partials per chunk
    constexpr int LPC = ChunkLanes<NPART, PPC>::LPC;       // lanes per chunk in chunk_totals
    constexpr int LUSED = ChunkLanes<NPART, PPC>::LUSED;   // lanes with distinct chunk totals
    constexpr int CPT = TILE / C;               // chunks per tile
    constexpr int SG = GradBytes<GK>::value;
    // in-kernel gradients drawn by dedicated warps (see draw_gradients)
    constexpr bool DRAW = GK == kGradPhilox && NDRAW > 0;
    constexpr int GKC = DRAW ? kGradF32 : GK;   // how the compressing threads read gradients
    // The 512 x 2 tile with stored gradients at C = 4096 (BERT-Large) is the
    // one instantiation where the options below measured slower.
    constexpr bool WIDE4096 = NT == 512 && SLOTS == 2 && C == 4096 && GK != kGradPhilox;
    // Full tiles do their element-wise sums in packed pairs (f32x2.cuh; the
    // same bits as the scalar form): faster for BERT-Base (512 x 2, C =
    // 2048), bfloat16 errors, C = 8192 and in-kernel gradients (W = 32, 1-bit
    // LAMB: 52.90 -> 52.34 ms); 2 to 5 % slower for WIDE4096, with or
    // without spills.
    constexpr bool PACK = !WIDE4096;
    // The chunk scale's shortcut (chunk_scale) measured faster everywhere
    // but in WIDE4096 (3 % slower there), which keeps the plain division and
    // square root.
    constexpr bool FAST_SCALE = !WIDE4096;
    // 1-bit LAMB's server pass reads the frozen preconditioner and the old
    // fresh variance from the ring after its chunk-norm barrier instead of
    // holding them in registers across it, and releases those two slots at
    // the end of the tile.  It removes spills where registers are scarce
    // (three CTAs per SM at 80 registers, draw warps at 64) and measured
    // faster in every shape that uses it (same box, fused kernel: BERT-Large
    // with bfloat16 errors 8.55 -> 7.71 ms, W = 32 with in-kernel gradients
    // 54.15 -> 52.96 ms, BERT-Base 1.937 -> 1.917 ms, GPT-2-XL 24.01 -> 23.61
    // ms); in WIDE4096 it ran slower (11.11 against 10.92 ms).
    constexpr bool LATE = !ADAM && !WIDE4096;
    static_assert(NDRAW == 0 || GK == kGradPhilox, "draw warps only for in-kernel gradients");
    static_assert(TILE % C == 0, "a tile holds whole chunks");
    using R = Ring<TILE>;
    using SL = Stream<SG, ADAM>;
    extern __shared__ __align__(128) unsigned char ring[];
    __shared__ uint64_t full[NSLOT];
    __shared__ uint64_t gfull[DRAW ? kDrawSlots : 1], gempty[DRAW ? kDrawSlots : 1];
    __shared__ int stop_draw;
    __shared__ __align__(16) float red[2][NPART];
    __shared__ uint32_t lmax[kMaxChunkLayers];
    // gradient slots of the draw warps follow the copy ring
    float* const gring = reinterpret_cast<float*>(ring + (size_t)NSLOT * R::kSlot);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int W = P.W;
    const int TPC = SL::items(W);                       // stream items per tile
    // Wait bound of the main loop.  A shortened bound (fault injection) is
    // for the CTA that leaves a copy out; every other CTA keeps the default,
    // so heavy memory traffic cannot make it give up on a copy that is only
    // slow.
    const uint32_t tries = blockIdx.x == 0 ? P.wait_tries : kDefaultWaitTries;
    const int64_t ntiles = P.Np / TILE;
    const int64_t nloc = (ntiles - blockIdx.x + gridDim.x - 1) / gridDim.x;

    if (tid == 0) {
        for (int s = 0; s < NSLOT; ++s) tma::bar_init(&full[s], 1);
        if constexpr (DRAW) {
            for (int s = 0; s < kDrawSlots; ++s) {
                tma::bar_init(&gfull[s], NDRAW / 32);     // one arrival per warp
                tma::bar_init(&gempty[s], NT / 32);
            }
            stop_draw = 0;
        }
        tma::fence_init();
    }
    for (int i = tid; i < kMaxChunkLayers; i += NT) lmax[i] = 0u;
    __syncthreads();
    if constexpr (DRAW) {
        if (tid >= NT) {
            draw_gradients<TILE, NDRAW>(P, D, G, gring, gfull, gempty, nloc, &stop_draw);
            return;
        }
    }
    RingPos<kDrawSlots> gcp;                  // next gradient slot to read (DRAW)

    // ---- producer (thread 0): items in order, as long as all their slots
    // fit in the ring ahead of the released slot positions ------------------
    int issue_pos = 0, released = 0;          // slot positions (per CTA)
    int64_t issue_tile = 0;                   // local tile index of the next item
    int issue_r = 0;                          // its kind
    RingPos<NSLOT> ip;                        // its first slot
    auto issue_ready = [&]() {
        while (issue_tile < nloc) {
            const int n = SL::slots(issue_r, W);
            if (issue_pos + n > released + NSLOT) break;
            issue_item<TILE, SG, NSLOT, ADAM, EB>(blockIdx.x + issue_tile * gridDim.x, issue_r, ip,
                                                  issue_pos, P, D, G, ring, full);
            issue_pos += n;
            ip = ip.plus(n);
            if (++issue_r == TPC) { issue_r = 0; ++issue_tile; }
        }
    };
    if (tid == 0) issue_ready();
    RingPos<NSLOT> cp;                        // consumer: next slot to read

    bool bad = false;        // non-finite gradient seen
    bool lost = false;       // a stage wait gave up

    for (int64_t ti = 0; ti < nloc; ++ti) {
        const int64_t tile = blockIdx.x + ti * gridDim.x;
        const int64_t base = tile * TILE;
        const bool full_tile = base + TILE <= P.N;
        const int64_t k0 = base / C;                     // first chunk of the tile
        const int64_t klast = (k0 + CPT - 1 < P.K - 1) ? k0 + CPT - 1 : P.K - 1;
        const int l0 = D.chunk_l0[k0];
        // this lane's chunk in chunk_totals, and its element count
        const int lq = lane % LUSED;
        const int64_t kq = k0 + lq / LPC;
        const int64_t nq_raw = P.N - kq * C;
        const float nq = (float)(nq_raw >= C ? C : (nq_raw > 0 ? nq_raw : 0));
        const bool lane_stores_scale = lane < LUSED && (lq % LPC) == 0 && kq < P.K;

        int nv[SLOTS];
        int qsrc[SLOTS];       // lane holding the scale of this slot's chunk
#pragma unroll
        for (int s = 0; s < SLOTS; ++s) {
            const int64_t r = P.N - (base + s * NT * 4 + tid * 4);
            nv[s] = r >= 4 ? 4 : (r > 0 ? (int)r : 0);
            qsrc[s] = ((s * NT * 4 + warp * 128) / C) * LPC;
        }

        // in-kernel gradients: per-element std and Student-t flags
        float stdv[SLOTS][4];
        uint32_t heavy[SLOTS];
        if constexpr (GK == kGradPhilox && !DRAW) {
            int l = l0;
            int64_t lend = D.layer_end[l];
#pragma unroll
            for (int s = 0; s < SLOTS; ++s) {
                heavy[s] = 0u;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    stdv[s][c] = 0.0f;
                    if (c < nv[s]) {
                        const int64_t i = base + s * NT * 4 + tid * 4 + c;
                        while (i >= lend) { ++l; lend = D.layer_end[l]; }
                        stdv[s][c] = G.layer_std[l];
                        if (G.layer_heavy && G.layer_heavy[l]) heavy[s] |= 1u << c;
                    }
                }
            }
        }
        // this thread's elements all draw from one kind of stream (true
        // except at a boundary between a normal and a heavy-tailed tensor)
        bool all_normal = true, all_heavy = true;
        if constexpr (GK == kGradPhilox && !DRAW) {
#pragma unroll
            for (int s = 0; s < SLOTS; ++s) {
                all_normal = all_normal && heavy[s] == 0u;
                all_heavy = all_heavy && heavy[s] == 0xFu;
            }
        }

        // ---- item M: beta1 * m_old, kept for the whole tile ------------------
        // m_old is the dense momentum after the warmup, afterwards the last
        // step's server signs times its chunk scales (exactly the same values)
        float bm[SLOTS][4], acc[SLOTS][4];
        {
            if (!wait_slots<NSLOT>(full, cp, 1, tries)) lost = true;
            const unsigned char* a = ring + (uint32_t)cp.slot * R::kSlot;
            cp = cp.plus(1);
            if (P.m_packed) {
                const uint32_t* words = reinterpret_cast<const uint32_t*>(a);
                const float* scales = reinterpret_cast<const float*>(a + TILE / 8) + (k0 & 3);
#pragma unroll
                for (int s = 0; s < SLOTS; ++s) {
                    const int e0 = s * NT * 4 + tid * 4;
                    const uint32_t bits = words[e0 >> 5] >> (e0 & 31);
                    const float sc = scales[e0 / C];
#pragma unroll
                    for (int c = 0; c < 4; ++c) bm[s][c] = fmul(P.beta1, ((bits >> c) & 1u) ? sc : -sc);
                }
            } else {
#pragma unroll
                for (int s = 0; s < SLOTS; ++s) {
                    const float4 mo = *reinterpret_cast<const float4*>(a + (s * NT * 4 + tid * 4) * 4);
                    bm[s][0] = fmul(P.beta1, mo.x); bm[s][1] = fmul(P.beta1, mo.y);
                    bm[s][2] = fmul(P.beta1, mo.z); bm[s][3] = fmul(P.beta1, mo.w);
                }
            }
#pragma unroll
            for (int s = 0; s < SLOTS; ++s)
#pragma unroll
                for (int c = 0; c < 4; ++c) acc[s][c] = 0.0f;
        }

        // ---- phase 1: every worker compresses its chunks ----------------------
        for (int w = 0; w < W; ++w) {
            if (!wait_slots<NSLOT>(full, cp, SL::kPerWorker, tries)) lost = true;
            const unsigned char* a = ring + (uint32_t)cp.slot * R::kSlot;
            const void* eb = ring + (uint32_t)cp.plus(SL::kPerWorker - 1).slot * R::kSlot;
            cp = cp.plus(SL::kPerWorker);
            if constexpr (DRAW) {
                // this worker's gradients, written by the draw warps
                if (!wait_handoff(&gfull[gcp.slot], gcp.phase, nullptr)) lost = true;
                a = reinterpret_cast<const unsigned char*>(gring + gcp.slot * TILE);
            }
            float z[SLOTS][4];
            // in-kernel gradients.  Normal elements: the draws of all slots
            // as independent Philox chains (instruction-level parallelism).
            // Heavy-tailed elements: one Student-t draw each, again as
            // independent chains when all of the thread's elements are heavy.
            float gin[SLOTS][4];
            if constexpr (GK == kGradPhilox && !DRAW) {
                if (all_heavy) {
#pragma unroll
                    for (int s = 0; s < SLOTS; ++s)
#pragma unroll
                        for (int c = 0; c < 4; ++c)
                            gin[s][c] = fmul(G.heavy_scale,
                                             gen::student_t3(G.seed, base + s * NT * 4 + tid * 4 + c,
                                                             G.t, (uint32_t)w));
                } else {
#pragma unroll
                    for (int s = 0; s < SLOTS; ++s) {
                        gen::grads_normal4(G.seed, (uint64_t)(base + s * NT * 4 + tid * 4) >> 2, G.t,
                                           (uint32_t)w, gin[s]);
#pragma unroll
                        for (int c = 0; c < 4; ++c) gin[s][c] = fmul(stdv[s][c], gin[s][c]);
                    }
                    if (!all_normal) {
#pragma unroll
                        for (int s = 0; s < SLOTS; ++s) {
                            if (heavy[s]) {
#pragma unroll
                                for (int c = 0; c < 4; ++c)
                                    if ((heavy[s] >> c) & 1u)
                                        gin[s][c] = fmul(G.heavy_scale,
                                                         gen::student_t3(G.seed, base + s * NT * 4 + tid * 4 + c,
                                                                         G.t, (uint32_t)w));
                            }
                        }
                    }
                }
            }
            // Per-element work, specialised at compile time for tiles whose
            // elements all exist (every tile but the last): no validity logic.
            if (P.check_finite) {
#pragma unroll
                for (int s = 0; s < SLOTS; ++s) {
                    const int off = s * NT * 4 + tid * 4;
                    float g[4];
                    load_grad4<GKC>(a, off, gin[s], g);
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        if (c < nv[s] && !isfinite(g[c])) bad = true;
                }
            }
            auto momentum_and_norms = [&](auto full_c) {
                constexpr bool FULL = decltype(full_c)::value;
                float part[SLOTS];
#pragma unroll
                for (int s = 0; s < SLOTS; ++s) {
                    const int off = s * NT * 4 + tid * 4;
                    float g[4], ee[4];
                    load_grad4<GKC>(a, off, gin[s], g);
                    load_err4<EB>(eb, off, ee);
                    if constexpr (FULL && PACK) {      // as below, the sums in packed pairs
                        float t[4];
#pragma unroll
                        for (int c = 0; c < 4; ++c) t[c] = fmul(P.omega1, g[c]);
                        add4(t, bm[s], t);
                        add4(z[s], t, ee);
                    } else {
#pragma unroll
                        for (int c = 0; c < 4; ++c) {
                            const float mw = fadd(bm[s][c], fmul(P.omega1, g[c]));
                            z[s][c] = (FULL || c < nv[s]) ? fadd(mw, ee[c]) : 0.0f;
                        }
                    }
                    if constexpr (PACK) {
                        float q[4];
                        mul4(q, z[s], z[s]);
                        part[s] = fadd(fadd(q[0], q[1]), fadd(q[2], q[3]));
                    } else {
                        part[s] = fadd(fadd(fmul(z[s][0], z[s][0]), fmul(z[s][1], z[s][1])),
                                       fadd(fmul(z[s][2], z[s][2]), fmul(z[s][3], z[s][3])));
                    }
                }
                const float t = warp_trees128<SLOTS>(part, lane);
                if (lane < SLOTS) red[w & 1][tree_block<SLOTS>(lane) * NWARP + warp] = t;
            };
            if (full_tile) momentum_and_norms(std::true_type{});
            else momentum_and_norms(std::false_type{});
            if constexpr (DRAW) {
                // every gradient of the slot has been read: hand it back
                warp_arrive(&gempty[gcp.slot]);
                gcp = gcp.plus(1);
            }
            if (sync_or<NT, DRAW>(lost)) goto abort;
            released += (w == 0) ? 1 + SL::kPerWorker : SL::kPerWorker;
            if (tid == 0) issue_ready();
            const float Sq = chunk_totals<NPART, PPC>(red[w & 1], lane);
            const float sq = chunk_scale<C, FAST_SCALE>(Sq, nq);
            // this thread's error elements, and the sign words its lane stores
            const int64_t eoff = (int64_t)w * P.Np + base + tid * 4;
            uint32_t* sw = D.signs_w + (int64_t)w * P.words_ld + (base + warp * 128) / 32 + (lane >> 3);
            auto signs_and_errors = [&](auto full_c) {
                constexpr bool FULL = decltype(full_c)::value;
                uint32_t nib[SLOTS];
#pragma unroll
                for (int s = 0; s < SLOTS; ++s) {
                    const float sc = (CPT == 1) ? sq : __shfl_sync(0xFFFFFFFFu, sq, qsrc[s]);
                    const float nsc = -sc;
                    float en[4], ssv[4];
                    nib[s] = 0u;
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const bool valid = FULL || c < nv[s];
                        const bool neg = z[s][c] < 0.0f;       // +0, -0 and NaN send +1
                        ssv[c] = neg ? nsc : sc;
                        if (!neg && valid) nib[s] |= 1u << c;
                    }
                    if constexpr (FULL && PACK) {
                        sub4(en, z[s], ssv);
                    } else {
#pragma unroll
                        for (int c = 0; c < 4; ++c) en[c] = (FULL || c < nv[s]) ? fsub(z[s][c], ssv[c]) : 0.0f;
                    }
                    if constexpr (PACK) {
                        add4(acc[s], acc[s], ssv);
                    } else {
#pragma unroll
                        for (int c = 0; c < 4; ++c) acc[s][c] = fadd(acc[s][c], ssv[c]);
                    }
                    store_err4<EB>(D.e_w, eoff + s * NT * 4, en);
                }
                const uint32_t word = pack_words<SLOTS>(nib, lane);
                if ((lane & 7) < SLOTS) sw[tree_block<SLOTS>(lane) * (NT * 4 / 32)] = word;
            };
            if (full_tile) signs_and_errors(std::true_type{});
            else signs_and_errors(std::false_type{});
            if (warp == 0 && lane_stores_scale) D.scale_w[(int64_t)w * P.K + kq] = sq;
        }

        // ---- phases 2 and 3: server average, recompression, scatter ----------
        {
            const int nsrv = SL::kServer + (ADAM ? 0 : 1);      // S (and F) slots
            if (!wait_slots<NSLOT>(full, cp, nsrv, tries)) lost = true;
            const float* es_in = reinterpret_cast<const float*>(ring + (uint32_t)cp.slot * R::kSlot);
            const float* d_in = reinterpret_cast<const float*>(ring + (uint32_t)cp.plus(1).slot * R::kSlot);
            const float* vf_in = reinterpret_cast<const float*>(ring + (uint32_t)cp.plus(2).slot * R::kSlot);
            cp = cp.plus(nsrv);
            float y[SLOTS][4], dz[SLOTS][4], vfo[SLOTS][4];
            auto average_and_norms = [&](auto full_c) {
                constexpr bool FULL = decltype(full_c)::value;
                float part[SLOTS];
#pragma unroll
                for (int s = 0; s < SLOTS; ++s) {
                    const int off = s * NT * 4 + tid * 4;
                    float ee[4];
                    load_err4<EB>(es_in, off, ee);
                    if constexpr (!ADAM && !LATE) {
                        const float4 v = *reinterpret_cast<const float4*>(d_in + off);
                        const float4 f = *reinterpret_cast<const float4*>(vf_in + off);
                        dz[s][0] = v.x; dz[s][1] = v.y; dz[s][2] = v.z; dz[s][3] = v.w;
                        vfo[s][0] = f.x; vfo[s][1] = f.y; vfo[s][2] = f.z; vfo[s][3] = f.w;
                    }
                    if constexpr (FULL && PACK) {      // the sums in packed pairs
                        float t[4];
#pragma unroll
                        for (int c = 0; c < 4; ++c) t[c] = div_w(acc[s][c], P);
                        add4(y[s], t, ee);
                    } else {
#pragma unroll
                        for (int c = 0; c < 4; ++c)
                            y[s][c] = (FULL || c < nv[s]) ? fadd(div_w(acc[s][c], P), ee[c]) : 0.0f;
                    }
                    if constexpr (PACK) {
                        float q[4];
                        mul4(q, y[s], y[s]);
                        part[s] = fadd(fadd(q[0], q[1]), fadd(q[2], q[3]));
                    } else {
                        part[s] = fadd(fadd(fmul(y[s][0], y[s][0]), fmul(y[s][1], y[s][1])),
                                       fadd(fmul(y[s][2], y[s][2]), fmul(y[s][3], y[s][3])));
                    }
                }
                const float t = warp_trees128<SLOTS>(part, lane);
                if (lane < SLOTS) red[W & 1][tree_block<SLOTS>(lane) * NWARP + warp] = t;
            };
            if (full_tile) average_and_norms(std::true_type{});
            else average_and_norms(std::false_type{});
            if (sync_or<NT, DRAW>(lost)) goto abort;
            released += LATE ? 1 : nsrv;
            if (tid == 0) issue_ready();
            const float SSq = chunk_totals<NPART, PPC>(red[W & 1], lane);
            const float ssq = chunk_scale<C, FAST_SCALE>(SSq, nq);

            // Per-tensor max of rho: a running max per thread, flushed into the
            // tile's shared per-tensor slots (or global, past kMaxChunkLayers)
            // whenever the tensor changes.  A full tile inside one tensor needs
            // no per-element tensor tracking.
            int l = l0;
            int64_t lend = D.layer_end[l];
            const bool one_tensor = full_tile && lend >= base + TILE;
            int lcur = -1;
            uint32_t runmax = 0u;
            auto flush_max = [&]() {
                if (lcur >= 0) {
                    if (lcur - l0 < kMaxChunkLayers) atomicMax(&lmax[lcur - l0], runmax);
                    else atomicMax(&D.Rmax[lcur], runmax);
                }
            };
            auto recompress_and_scatter = [&](auto full_c, auto one_c) {
                constexpr bool FULL = decltype(full_c)::value;
                constexpr bool ONE = decltype(one_c)::value;
                if constexpr (ONE && !ADAM) lcur = l0;
                uint32_t nib[SLOTS];
#pragma unroll
                for (int s = 0; s < SLOTS; ++s) {
                    const int off = s * NT * 4 + tid * 4;
                    const float ss = (CPT == 1) ? ssq : __shfl_sync(0xFFFFFFFFu, ssq, qsrc[s]);
                    const float nss = -ss;
                    float es[4], mn[4], vf[4], den[4];
                    nib[s] = 0u;
                    if constexpr (LATE) {
                        const float4 v = *reinterpret_cast<const float4*>(d_in + off);
                        const float4 f = *reinterpret_cast<const float4*>(vf_in + off);
                        dz[s][0] = v.x; dz[s][1] = v.y; dz[s][2] = v.z; dz[s][3] = v.w;
                        vfo[s][0] = f.x; vfo[s][1] = f.y; vfo[s][2] = f.z; vfo[s][3] = f.w;
                    }
                    constexpr bool PK = FULL && PACK;
                    if constexpr (PK) {
                        // the per-element formulas below, in packed pairs
#pragma unroll
                        for (int c = 0; c < 4; ++c) {
                            const bool neg = y[s][c] < 0.0f;
                            mn[c] = neg ? nss : ss;
                            if (!neg) nib[s] |= 1u << c;
                        }
                        sub4(es, y[s], mn);
                        if constexpr (!ADAM) {
                            float dm[4], gt[4], t1[4], t2[4];
                            sub4(dm, mn, bm[s]);
#pragma unroll
                            for (int c = 0; c < 4; ++c) gt[c] = fdiv(dm[c], P.omega1);
                            mul4(t1, gt, gt);
                            mul4s(t1, P.omega2, t1);
                            mul4s(t2, P.beta2, vfo[s]);
#pragma unroll
                            for (int c = 0; c < 4; ++c) vf[c] = fadd(t2[c], t1[c]);   // products: scalar sums
#pragma unroll
                            for (int c = 0; c < 4; ++c) t1[c] = fsqrt(vf[c]);
                            add4s(den, t1, P.eps);
                        }
                    }
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const bool valid = FULL || c < nv[s];
                        if constexpr (!PK) {
                            const bool neg = y[s][c] < 0.0f;
                            const float sgn = neg ? nss : ss;
                            if (!neg && valid) nib[s] |= 1u << c;
                            es[c] = valid ? fsub(y[s][c], sgn) : 0.0f;
                            mn[c] = valid ? sgn : 0.0f;
                        }
                        if constexpr (ADAM) continue;
                        if constexpr (!PK) {
                            // reconstructed gradient and fresh second moment
                            const float gt = fdiv(fsub(mn[c], bm[s][c]), P.omega1);
                            vf[c] = valid ? fadd(fmul(P.beta2, vfo[s][c]), fmul(P.omega2, fmul(gt, gt))) : 0.0f;
                            den[c] = fadd(fsqrt(vf[c]), P.eps);
                        }
                        if (valid) {
                            float rho = fdiv(dz[s][c], den[c]);
                            if (rho != rho) rho = __int_as_float(0x7F800000);
                            if constexpr (!ONE) {
                                const int64_t i = base + off + c;
                                while (i >= lend) { ++l; lend = D.layer_end[l]; }
                                if (l != lcur) {
                                    flush_max();
                                    lcur = l;
                                    runmax = 0u;
                                }
                            }
                            runmax = max(runmax, __float_as_uint(rho));
                        }
                    }
                    store_err4<EB>(D.e_s, base + off, es);
                    if constexpr (!ADAM)
                        *reinterpret_cast<float4*>(D.v_fresh + base + off) =
                            make_float4(vf[0], vf[1], vf[2], vf[3]);
                }
                const uint32_t word = pack_words<SLOTS>(nib, lane);
                if ((lane & 7) < SLOTS)
                    D.signs_s[(base + warp * 128) / 32 + (lane >> 3) + tree_block<SLOTS>(lane) * (NT * 4 / 32)] = word;
            };
            if (one_tensor) recompress_and_scatter(std::true_type{}, std::true_type{});
            else if (full_tile) recompress_and_scatter(std::true_type{}, std::false_type{});
            else recompress_and_scatter(std::false_type{}, std::false_type{});
            flush_max();
            if (warp == 0 && lane_stores_scale) D.scale_s[kq] = ssq;
        }
        sync_all<NT, DRAW>();
        if constexpr (LATE) {                      // the server's last two slots
            released += 2;
            if (tid == 0) issue_ready();
        }
        {
            const int nl = D.chunk_l1[klast] - l0 + 1;
            for (int jj = tid; jj < nl && jj < kMaxChunkLayers; jj += NT) {
                const uint32_t v = lmax[jj];
                lmax[jj] = 0u;
                if (v) atomicMax(&D.Rmax[l0 + jj], v);
            }
        }
    }
    if (bad) atomicOr(D.flags, 1u);
    return;

abort:
    // A stage wait gave up (never expected).  Record it, let the copies this
    // CTA still has in flight land (bounded), then leave.
    if (tid == 0) {
        atomicOr(D.flags, 2u);
        if constexpr (DRAW) *(volatile int*)&stop_draw = 1;     // the draw warps leave too
        // every slot position issued but not yet released (at most NSLOT):
        // they end at the producer's position ip.  Each one whose copies were
        // issued is waited for with the default bound, whatever bound the
        // main loop used, so that no bulk copy is still writing into this
        // CTA's shared memory when it exits; only the position that fault
        // injection left out (nothing in flight there) is passed over.
        RingPos<NSLOT> q = ip;
        for (int pnum = issue_pos - 1; pnum >= released; --pnum) {
            q.slot -= 1;
            if (q.slot < 0) { q.slot += NSLOT; q.phase ^= 1u; }
            if (blockIdx.x == 0 && pnum == P.skip_copy) continue;
            wait_stage(&full[q.slot], q.phase, kDefaultWaitTries);
        }
    }
    sync_all<NT, DRAW>();
}

cudaError_t launch_update(const Problem& P, const Dev& D, float* x, int msig, cudaStream_t st);

template <int NT, int SLOTS, int GK, int NSLOT, int C, bool ADAM, bool EB, int NDRAW = 0>
static cudaError_t launch_one(const Problem& P, const Dev& D, const Grads& G, cudaStream_t st)
{
    constexpr int TILE = NT * 4 * SLOTS;
    // the copy ring, then (with draw warps) the gradient slots
    constexpr size_t smem = (size_t)NSLOT * Ring<TILE>::kSlot
                            + (NDRAW > 0 ? (size_t)kDrawSlots * TILE * 4 : 0);
    auto kern = k_compress<NT, SLOTS, GK, NSLOT, C, ADAM, EB, NDRAW>;
    // Launch shape per device and instantiation, set up on first use.  A slot
    // is published only after its device's function attributes are set, and
    // concurrent first uses on one device just repeat the same settings, so
    // host threads driving different GPUs need no lock.
    constexpr int kCachedDevices = 64;
    static std::atomic<int> grid_cap_of[kCachedDevices];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    int grid_cap = dev < kCachedDevices ? grid_cap_of[dev].load(std::memory_order_acquire) : 0;
    if (grid_cap == 0) {
        if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)))
            return e;
        if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                                      cudaSharedmemCarveoutMaxShared)))
            return e;
        int per_sm = 0, sms = 0;
        if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, NT + NDRAW, smem))) return e;
        if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev))) return e;
        grid_cap = (per_sm > 0 ? per_sm : 1) * sms;
        if (dev < kCachedDevices) grid_cap_of[dev].store(grid_cap, std::memory_order_release);
    }
    const int64_t ntiles = P.Np / TILE;
    const unsigned grid = (unsigned)(ntiles < grid_cap ? ntiles : grid_cap);
    kern<<<grid, NT + NDRAW, smem, st>>>(P, D, G);
    return cudaGetLastError();
}

template <int NT, int SLOTS, int NSLOT, int C, bool ADAM, bool EB>
static cudaError_t launch_grad(const Problem& P, const Dev& D, const Grads& G, cudaStream_t st)
{
    switch (G.kind) {
    case kGradF32:  return launch_one<NT, SLOTS, kGradF32, NSLOT, C, ADAM, EB>(P, D, G, st);
    case kGradBF16: return launch_one<NT, SLOTS, kGradBF16, NSLOT, C, ADAM, EB>(P, D, G, st);
    default:        return launch_one<NT, SLOTS, kGradPhilox, NSLOT, C, ADAM, EB>(P, D, G, st);
    }
}

// One translation unit per (variant, error storage) instantiates this for
// every chunk size; see k_compress_*.cu.
template <bool ADAM, bool EB>
cudaError_t launch_fused(const Problem& P, const Dev& D, const Grads& G, cudaStream_t st);

template <bool ADAM, bool EB>
cudaError_t launch_fused_all_chunks(const Problem& P, const Dev& D, const Grads& G, cudaStream_t st)
{
    // 4096-element tiles (256 threads x 4 float4 groups) holding 4096/C chunks;
    // 8192-element chunks use 512-thread tiles of one chunk.  For C = 2048 and
    // 4096 with stored binary32 gradients and errors (streaming-bound cases)
    // the same tile is split over 512 threads x 2 groups: 64 registers, so
    // two CTAs give 32 warps per SM to cover the arithmetic between the
    // barriers (same-box A/B, fused kernel: BERT-Large 11.72 -> 11.22 ms,
    // BERT-Base 2.05 -> 1.99 ms).  With bfloat16 errors the wider CTA runs
    // 23 % slower, so those keep 256 threads, and at C = 4096 run three CTAs
    // per SM with a 4-slot ring (1-bit LAMB reading its server inputs late:
    // BERT-Large fused kernel 8.55 -> 7.71 ms, same box).  1-bit Adam with
    // binary32 errors at C = 4096 takes the same three-CTA shape (10.79 ->
    // 10.54 ms); 1-bit LAMB there spills at its 80 registers and keeps the
    // 512-thread tile (11.06 against 11.22 ms).  In-kernel gradients at
    // C = 4096 add 512 draw threads (draw_gradients).
    switch (P.C) {
    case 256:  return launch_grad<256, 4, 7, 256, ADAM, EB>(P, D, G, st);
    case 512:  return launch_grad<256, 4, 7, 512, ADAM, EB>(P, D, G, st);
    case 1024: return launch_grad<256, 4, 7, 1024, ADAM, EB>(P, D, G, st);
    case 2048:
        if constexpr (!EB)
            if (G.kind == kGradF32) return launch_one<512, 2, kGradF32, 7, 2048, ADAM, EB>(P, D, G, st);
        return launch_grad<256, 4, 7, 2048, ADAM, EB>(P, D, G, st);
    case 4096:
        if (G.kind == kGradPhilox) return launch_one<512, 2, kGradPhilox, 7, 4096, ADAM, EB, 512>(P, D, G, st);
        if (G.kind == kGradF32) {
            if constexpr (ADAM || EB)   // three CTAs per SM with a 4-slot ring
                return launch_one<256, 4, kGradF32, 4, 4096, ADAM, EB>(P, D, G, st);
            else
                return launch_one<512, 2, kGradF32, 7, 4096, ADAM, EB>(P, D, G, st);
        }
        return launch_grad<256, 4, 7, 4096, ADAM, EB>(P, D, G, st);
    case 8192: return launch_grad<512, 4, 7, 8192, ADAM, EB>(P, D, G, st);
    default:   return cudaErrorInvalidValue;
    }
}

}  // namespace lamb1b
