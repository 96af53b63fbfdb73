// Host side of the lamb1b C ABI (include/lamb1b.h): argument validation, the
// workspace layout, the stage state machine and the kernel launches.
#include <cmath>
#include <cstdint>
#include <cstring>
#include <new>
#include <vector>

#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include "lamb1b.h"
#include "lamb1b_internal.cuh"
#include "device_ptr.h"

using lamb1b::Dev;
using lamb1b::Grads;
using lamb1b::Problem;

namespace {

enum Region {
    R_M, R_V, R_VF, R_DF, R_ES, R_EW, R_SW, R_SS, R_SCW, R_SCS,
    R_CBAR, R_RPREV, R_CCUR, R_GC, R_RLAST, R_SX, R_SU, R_RMAX,
    R_LOFF, R_LEND, R_HBASE, R_CL0, R_CL1, R_PX, R_PU, R_BBASE, R_BX, R_BU, R_FLAGS, R_COUNT
};

struct Plan {
    int64_t N = 0, Np = 0, K = 0, words_ld = 0, H = 0, NB = 0;
    int32_t L = 0, W = 0, C = 0;
    size_t off[R_COUNT] = {};
    size_t total = 0;
};

bool finite(float v) { return std::isfinite(v); }

int check_hparams(const lamb1b_hparams* hp)
{
    if (!hp) return LAMB1B_ERR_ARG;
    if (hp->W < 1 || hp->W > 256) return LAMB1B_ERR_ARG;
    const int C = hp->chunk;
    if (C < 256 || C > 8192 || (C & (C - 1))) return LAMB1B_ERR_ARG;
    const float f[] = {hp->lr, hp->beta1, hp->beta2, hp->eps, hp->weight_decay, hp->coeff_min,
                       hp->coeff_max, hp->coeff_ema, hp->factor_min, hp->factor_max,
                       hp->factor_threshold};
    for (float v : f)
        if (!finite(v)) return LAMB1B_ERR_ARG;
    if (!(hp->beta1 >= 0.0f && hp->beta1 < 1.0f)) return LAMB1B_ERR_ARG;
    if (!(hp->beta2 >= 0.0f && hp->beta2 <= 1.0f)) return LAMB1B_ERR_ARG;
    if (!(hp->eps >= 0.0f)) return LAMB1B_ERR_ARG;
    if (!(hp->coeff_min >= 0.0f && hp->coeff_min <= hp->coeff_max)) return LAMB1B_ERR_ARG;
    if (!(hp->coeff_ema >= 0.0f && hp->coeff_ema <= 1.0f)) return LAMB1B_ERR_ARG;
    if (!(hp->factor_min >= 0.0f && hp->factor_min <= hp->factor_max)) return LAMB1B_ERR_ARG;
    if (!(hp->factor_threshold >= 0.0f)) return LAMB1B_ERR_ARG;
    if (hp->check_finite != 0 && hp->check_finite != 1) return LAMB1B_ERR_ARG;
    if (hp->variant != 0 && hp->variant != 1) return LAMB1B_ERR_ARG;
    if (hp->error_storage != 0 && hp->error_storage != 1) return LAMB1B_ERR_ARG;
    return LAMB1B_OK;
}

int make_plan(const lamb1b_layer* layers, int32_t L, const lamb1b_hparams* hp, Plan* p)
{
    int rc = check_hparams(hp);
    if (rc) return rc;
    if (!layers || L < 1 || L > (1 << 24)) return LAMB1B_ERR_ARG;
    int64_t N = 0, H = 0, NB = 0;
    for (int32_t l = 0; l < L; ++l) {
        if (layers[l].offset != N || layers[l].numel < 1) return LAMB1B_ERR_ARG;
        if (layers[l].numel > (int64_t(1) << 40) - N) return LAMB1B_ERR_ARG;
        const int64_t g0 = layers[l].offset / lamb1b::kGranule;
        const int64_t g1 = (layers[l].offset + layers[l].numel - 1) / lamb1b::kGranule;
        H += 2 * (g1 - g0 + 1);
        NB += lamb1b::level1_blocks(g1 - g0 + 1);
        N += layers[l].numel;
    }
    if (NB > 0x7FFFFFFFll) return LAMB1B_ERR_ARG;
    p->N = N;
    p->L = L;
    p->W = hp->W;
    p->C = hp->chunk;
    p->K = (N + p->C - 1) / p->C;
    if (p->K > 0x7FFFFFFFll) return LAMB1B_ERR_ARG;
    p->Np = lamb1b::padded_length(N, p->C);   // whole compression tiles
    p->words_ld = p->Np / 32;
    p->H = H;
    p->NB = NB;
    const size_t f = sizeof(float);
    size_t bytes[R_COUNT];
    const size_t fe = hp->error_storage ? 2 : 4;   // error element size
    bytes[R_M] = bytes[R_V] = bytes[R_VF] = bytes[R_DF] = f * p->Np;
    bytes[R_ES] = fe * p->Np;
    bytes[R_EW] = fe * p->Np * p->W;
    bytes[R_SW] = sizeof(uint32_t) * p->words_ld * p->W;
    bytes[R_SS] = sizeof(uint32_t) * p->words_ld;
    bytes[R_SCW] = f * p->K * p->W;
    bytes[R_SCS] = f * (p->K + 16);   // + room for 16-byte aligned windows
    for (int r = R_CBAR; r <= R_RMAX; ++r) bytes[r] = f * L;
    bytes[R_LOFF] = bytes[R_LEND] = sizeof(int64_t) * L;
    bytes[R_HBASE] = sizeof(int64_t) * (L + 1);
    bytes[R_CL0] = bytes[R_CL1] = sizeof(int32_t) * p->K;
    bytes[R_PX] = bytes[R_PU] = f * H;
    bytes[R_BBASE] = sizeof(int64_t) * (L + 1);
    bytes[R_BX] = bytes[R_BU] = f * NB;
    bytes[R_FLAGS] = 16;
    size_t cur = 0;
    for (int r = 0; r < R_COUNT; ++r) {
        p->off[r] = cur;
        cur = (cur + bytes[r] + 255) & ~size_t(255);
    }
    p->total = cur;
    return LAMB1B_OK;
}

int grads_check(const lamb1b_ctx* ctx, const lamb1b_grads* g);
using lamb1b::is_device_ptr;

// NVTX range around the host side of one stage (enqueue only), so profiler
// timelines show which library call launched which kernels.
struct NvtxRange {
    explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
};

}  // namespace

struct lamb1b_ctx {
    int device = 0;
    Problem P{};
    Dev D{};
    float* x = nullptr;
    int64_t t = 0;
    int32_t n_warm = 0;
    int32_t stage = 0;
    std::vector<int64_t> off, end, hbase, bbase;
    std::vector<int32_t> l0, l1;
    bool tracing = false;
    bool d_frz_valid = false;   // D.d_frz holds sqrt(v) + eps of the frozen v
    cudaEvent_t ev[4] = {};
    // lamb1b_compress_step_host: the staging buffers seen lately, each with
    // an event recorded after the last step that read it, so that the next
    // copy into it waits for that step only
    struct Staging {
        const void* ptr = nullptr;
        cudaEvent_t used = nullptr;
        bool recorded = false;
        uint64_t last = 0;
    };
    static constexpr int kStaging = 4;
    Staging stg[kStaging];
    uint64_t stg_clock = 0;
    cudaEvent_t copied = nullptr;   // the host-to-device copy of a step is done
    cudaEvent_t fence = nullptr;    // all work enqueued on the step stream so far

    ~lamb1b_ctx()
    {
        for (Staging& e : stg)
            if (e.used) cudaEventDestroy(e.used);
        if (copied) cudaEventDestroy(copied);
        if (fence) cudaEventDestroy(fence);
    }
};

namespace {

int grads_check(const lamb1b_ctx* ctx, const lamb1b_grads* g)
{
    if (!g) return LAMB1B_ERR_ARG;
    if (ctx->t > 0xFFFFFFFFll) return LAMB1B_ERR_STATE;
    switch (g->kind) {
    case LAMB1B_GRAD_F32:
    case LAMB1B_GRAD_BF16: {
        const int64_t es = g->kind == LAMB1B_GRAD_F32 ? 4 : 2;
        if (!g->ptr || g->ld < ctx->P.N) return LAMB1B_ERR_ARG;
        if ((reinterpret_cast<uintptr_t>(g->ptr) & 15u) || ((g->ld * es) & 15)) return LAMB1B_ERR_ALIGN;
        // the kernels stage gradients with bulk copies from this GPU's memory
        if (!is_device_ptr(g->ptr, ctx->device)) return LAMB1B_ERR_ARG;
        return LAMB1B_OK;
    }
    case LAMB1B_GRAD_PHILOX:
        if (!g->layer_std || !finite(g->heavy_scale)) return LAMB1B_ERR_ARG;
        if (!is_device_ptr(g->layer_std, ctx->device) ||
            (g->layer_heavy && !is_device_ptr(g->layer_heavy, ctx->device)))
            return LAMB1B_ERR_ARG;
        return LAMB1B_OK;
    default:
        return LAMB1B_ERR_ARG;
    }
}

Grads to_grads(const lamb1b_ctx* ctx, const lamb1b_grads* g)
{
    Grads G;
    G.kind = g->kind;
    G.ptr = g->ptr;
    G.ld = g->ld;
    G.seed = g->seed;
    G.layer_std = g->layer_std;
    G.layer_heavy = g->layer_heavy;
    G.heavy_scale = g->heavy_scale;
    G.t = (uint32_t)ctx->t;
    return G;
}

int device_check(const lamb1b_ctx* ctx)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return LAMB1B_ERR_CUDA;
    return dev == ctx->device ? LAMB1B_OK : LAMB1B_ERR_DEVICE;
}


}  // namespace

extern "C" size_t lamb1b_workspace_bytes(const lamb1b_layer* layers, int32_t L,
                                         const lamb1b_hparams* hp)
{
    Plan p;
    if (make_plan(layers, L, hp, &p) != LAMB1B_OK) return 0;
    return p.total;
}

extern "C" int lamb1b_init(lamb1b_ctx** out, const lamb1b_layer* layers, int32_t L,
                           const lamb1b_hparams* hp, float* params_dev, void* workspace_dev,
                           size_t workspace_bytes, void* stream)
{
    if (!out) return LAMB1B_ERR_ARG;
    *out = nullptr;
    Plan p;
    int rc = make_plan(layers, L, hp, &p);
    if (rc) return rc;
    if (!params_dev || !workspace_dev) return LAMB1B_ERR_ARG;
    if (reinterpret_cast<uintptr_t>(params_dev) & 15u) return LAMB1B_ERR_ALIGN;
    if (reinterpret_cast<uintptr_t>(workspace_dev) & 255u) return LAMB1B_ERR_ALIGN;
    if (workspace_bytes < p.total) return LAMB1B_ERR_WORKSPACE;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return LAMB1B_ERR_CUDA;
    if (!is_device_ptr(params_dev, dev) || !is_device_ptr(workspace_dev, dev)) return LAMB1B_ERR_ARG;

    lamb1b_ctx* c = new (std::nothrow) lamb1b_ctx();
    if (!c) return LAMB1B_ERR_ARG;
    c->device = dev;
    c->x = params_dev;

    Problem& P = c->P;
    P.N = p.N; P.Np = p.Np; P.K = p.K; P.words_ld = p.words_ld;
    P.L = p.L; P.W = p.W; P.C = p.C;
    P.lr = hp->lr; P.beta1 = hp->beta1; P.beta2 = hp->beta2; P.eps = hp->eps;
    P.wd = hp->weight_decay;
    P.omega1 = 1.0f - hp->beta1;     // one binary32 subtraction each
    P.omega2 = 1.0f - hp->beta2;
    P.cmin = hp->coeff_min; P.cmax = hp->coeff_max; P.cema = hp->coeff_ema;
    P.one_m_cema = 1.0f - hp->coeff_ema;
    P.fmin = hp->factor_min; P.fmax = hp->factor_max;
    P.fthr_lo = 1.0f - hp->factor_threshold;
    P.fthr_hi = 1.0f + hp->factor_threshold;
    P.check_finite = hp->check_finite;
    P.adam = hp->variant == 1 ? 1 : 0;
    P.ebf16 = hp->error_storage == 1 ? 1 : 0;
    P.wait_tries = lamb1b::kDefaultWaitTries;
    P.skip_copy = -1;
    P.log2c = 0;
    while ((1 << P.log2c) < p.C) ++P.log2c;
    P.w_pow2 = (p.W & (p.W - 1)) == 0 ? 1 : 0;
    P.inv_w = 1.0f / (float)p.W;

    char* ws = static_cast<char*>(workspace_dev);
    Dev& D = c->D;
    D.m = reinterpret_cast<float*>(ws + p.off[R_M]);
    D.v = reinterpret_cast<float*>(ws + p.off[R_V]);
    D.v_fresh = reinterpret_cast<float*>(ws + p.off[R_VF]);
    D.d_frz = reinterpret_cast<float*>(ws + p.off[R_DF]);
    D.e_s = reinterpret_cast<float*>(ws + p.off[R_ES]);
    D.e_w = reinterpret_cast<float*>(ws + p.off[R_EW]);
    D.signs_w = reinterpret_cast<uint32_t*>(ws + p.off[R_SW]);
    D.signs_s = reinterpret_cast<uint32_t*>(ws + p.off[R_SS]);
    D.scale_w = reinterpret_cast<float*>(ws + p.off[R_SCW]);
    D.scale_s = reinterpret_cast<float*>(ws + p.off[R_SCS]);
    D.c_bar = reinterpret_cast<float*>(ws + p.off[R_CBAR]);
    D.r_prev = reinterpret_cast<float*>(ws + p.off[R_RPREV]);
    D.c_cur = reinterpret_cast<float*>(ws + p.off[R_CCUR]);
    D.gc = reinterpret_cast<float*>(ws + p.off[R_GC]);
    D.R_last = reinterpret_cast<float*>(ws + p.off[R_RLAST]);
    D.Sx = reinterpret_cast<float*>(ws + p.off[R_SX]);
    D.Su = reinterpret_cast<float*>(ws + p.off[R_SU]);
    D.Rmax = reinterpret_cast<uint32_t*>(ws + p.off[R_RMAX]);
    D.layer_off = reinterpret_cast<int64_t*>(ws + p.off[R_LOFF]);
    D.layer_end = reinterpret_cast<int64_t*>(ws + p.off[R_LEND]);
    D.hbase = reinterpret_cast<int64_t*>(ws + p.off[R_HBASE]);
    D.chunk_l0 = reinterpret_cast<int32_t*>(ws + p.off[R_CL0]);
    D.chunk_l1 = reinterpret_cast<int32_t*>(ws + p.off[R_CL1]);
    D.part_x = reinterpret_cast<float*>(ws + p.off[R_PX]);
    D.part_u = reinterpret_cast<float*>(ws + p.off[R_PU]);
    D.bbase = reinterpret_cast<int64_t*>(ws + p.off[R_BBASE]);
    D.blk_x = reinterpret_cast<float*>(ws + p.off[R_BX]);
    D.blk_u = reinterpret_cast<float*>(ws + p.off[R_BU]);
    P.NB = p.NB;
    D.flags = reinterpret_cast<uint32_t*>(ws + p.off[R_FLAGS]);

    // host tables
    c->off.resize(L);
    c->end.resize(L);
    c->hbase.resize(L + 1);
    c->bbase.resize(L + 1);
    c->hbase[0] = 0;
    c->bbase[0] = 0;
    for (int32_t l = 0; l < L; ++l) {
        c->off[l] = layers[l].offset;
        c->end[l] = layers[l].offset + layers[l].numel;
        const int64_t g0 = c->off[l] / lamb1b::kGranule, g1 = (c->end[l] - 1) / lamb1b::kGranule;
        c->hbase[l + 1] = c->hbase[l] + 2 * (g1 - g0 + 1);
        c->bbase[l + 1] = c->bbase[l] + lamb1b::level1_blocks(g1 - g0 + 1);
    }
    c->l0.resize(p.K);
    c->l1.resize(p.K);
    int32_t l = 0;
    for (int64_t k = 0; k < p.K; ++k) {
        const int64_t first = k * p.C;
        const int64_t last = (first + p.C <= p.N ? first + p.C : p.N) - 1;
        while (c->end[l] <= first) ++l;
        c->l0[k] = l;
        int32_t m = l;
        while (c->end[m] <= last) ++m;
        c->l1[k] = m;
    }

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    bool ok = cudaMemsetAsync(workspace_dev, 0, p.total, st) == cudaSuccess;
    ok = ok && cudaMemcpyAsync(D.layer_off, c->off.data(), sizeof(int64_t) * L,
                               cudaMemcpyHostToDevice, st) == cudaSuccess;
    ok = ok && cudaMemcpyAsync(D.layer_end, c->end.data(), sizeof(int64_t) * L,
                               cudaMemcpyHostToDevice, st) == cudaSuccess;
    ok = ok && cudaMemcpyAsync(D.hbase, c->hbase.data(), sizeof(int64_t) * (L + 1),
                               cudaMemcpyHostToDevice, st) == cudaSuccess;
    ok = ok && cudaMemcpyAsync(D.bbase, c->bbase.data(), sizeof(int64_t) * (L + 1),
                               cudaMemcpyHostToDevice, st) == cudaSuccess;
    ok = ok && cudaMemcpyAsync(D.chunk_l0, c->l0.data(), sizeof(int32_t) * p.K,
                               cudaMemcpyHostToDevice, st) == cudaSuccess;
    ok = ok && cudaMemcpyAsync(D.chunk_l1, c->l1.data(), sizeof(int32_t) * p.K,
                               cudaMemcpyHostToDevice, st) == cudaSuccess;
    ok = ok && lamb1b::launch_init_layers(P, D, st) == cudaSuccess;
    // the host tables must outlive the copies: pageable copies are staged
    // before cudaMemcpyAsync returns, and the context keeps them anyway
    if (!ok) {
        cudaGetLastError();
        delete c;
        return LAMB1B_ERR_CUDA;
    }
    *out = c;
    return LAMB1B_OK;
}

extern "C" int lamb1b_warmup_step(lamb1b_ctx* ctx, const lamb1b_grads* grads, void* stream)
{
    if (!ctx) return LAMB1B_ERR_ARG;
    if (ctx->stage != 0) return LAMB1B_ERR_STATE;
    int rc = device_check(ctx);
    if (rc) return rc;
    if ((rc = grads_check(ctx, grads))) return rc;
    const Grads G = to_grads(ctx, grads);
    NvtxRange range("lamb1b warmup step");
    if (lamb1b::launch_warmup(ctx->P, ctx->D, G, ctx->x, static_cast<cudaStream_t>(stream),
                              ctx->n_warm == 0, ctx->tracing ? ctx->ev : nullptr) != cudaSuccess)
        return LAMB1B_ERR_CUDA;
    ctx->t += 1;
    ctx->n_warm += 1;
    return LAMB1B_OK;
}

extern "C" int lamb1b_freeze_variance(lamb1b_ctx* ctx, void* stream)
{
    if (!ctx) return LAMB1B_ERR_ARG;
    if (ctx->stage != 0) return LAMB1B_ERR_STATE;
    int rc = device_check(ctx);
    if (rc) return rc;
    NvtxRange range("lamb1b freeze variance");
    if (lamb1b::launch_freeze(ctx->P, ctx->D, static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return LAMB1B_ERR_CUDA;
    ctx->stage = 1;
    ctx->d_frz_valid = true;
    return LAMB1B_OK;
}

namespace {

// The kernels of one compression step on checked gradients.
int compress_enqueue(lamb1b_ctx* ctx, const lamb1b_grads* grads, cudaStream_t st)
{
    const Grads G = to_grads(ctx, grads);
    // after the first compression step m lives in the server's sign words
    // and chunk scales; before it, in the dense buffer the warmup left
    ctx->P.m_packed = ctx->t > ctx->n_warm ? 1 : 0;
    if (!ctx->d_frz_valid) {     // after a restore: rebuild sqrt(v) + eps of the frozen v
        if (lamb1b::launch_frozen_denominator(ctx->P, ctx->D, st) != cudaSuccess) return LAMB1B_ERR_CUDA;
        ctx->d_frz_valid = true;
    }
    if (lamb1b::launch_compress(ctx->P, ctx->D, G, ctx->x, st, ctx->tracing ? ctx->ev : nullptr) !=
        cudaSuccess)
        return LAMB1B_ERR_CUDA;
    ctx->t += 1;
    return LAMB1B_OK;
}

bool is_pinned_host_ptr(const void* p)
{
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return a.type == cudaMemoryTypeHost;
}

int refuse_capture(cudaStream_t st)
{
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(st, &cs) != cudaSuccess) {
        cudaGetLastError();
        return LAMB1B_ERR_CUDA;
    }
    return cs == cudaStreamCaptureStatusNone ? LAMB1B_OK : LAMB1B_ERR_ARG;
}

int make_event(cudaEvent_t* e)
{
    if (*e) return LAMB1B_OK;
    if (cudaEventCreateWithFlags(e, cudaEventDisableTiming) != cudaSuccess) {
        cudaGetLastError();
        *e = nullptr;
        return LAMB1B_ERR_CUDA;
    }
    return LAMB1B_OK;
}

}  // namespace

extern "C" int lamb1b_compress_step(lamb1b_ctx* ctx, const lamb1b_grads* grads, void* stream)
{
    if (!ctx) return LAMB1B_ERR_ARG;
    if (ctx->stage != 1) return LAMB1B_ERR_STATE;
    int rc = device_check(ctx);
    if (rc) return rc;
    if ((rc = grads_check(ctx, grads))) return rc;
    NvtxRange range("lamb1b compression step");
    return compress_enqueue(ctx, grads, static_cast<cudaStream_t>(stream));
}

extern "C" int lamb1b_compress_step_host(lamb1b_ctx* ctx, const lamb1b_grads* host_grads, void* staging,
                                         uint32_t* words_host, float* scales_host, void* stream,
                                         void* copy_stream)
{
    if (!ctx || !host_grads) return LAMB1B_ERR_ARG;
    if (ctx->stage != 1) return LAMB1B_ERR_STATE;
    int rc = device_check(ctx);
    if (rc) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaStream_t cst = static_cast<cudaStream_t>(copy_stream);
    // first, so that no pointer query runs inside a capture
    if ((rc = refuse_capture(st)) || (rc = refuse_capture(cst))) return rc;
    if (host_grads->kind != LAMB1B_GRAD_F32 && host_grads->kind != LAMB1B_GRAD_BF16) return LAMB1B_ERR_ARG;
    if (!host_grads->ptr || !is_pinned_host_ptr(host_grads->ptr)) return LAMB1B_ERR_ARG;
    if ((words_host && !is_pinned_host_ptr(words_host)) || (scales_host && !is_pinned_host_ptr(scales_host)))
        return LAMB1B_ERR_ARG;
    lamb1b_grads dev = *host_grads;      // the same rows, in the staging buffer
    dev.ptr = staging;
    if ((rc = grads_check(ctx, &dev))) return rc;
    if ((rc = make_event(&ctx->copied)) || (rc = make_event(&ctx->fence))) return rc;

    // the staging buffer's entry: the last step that read it, or (a buffer
    // not seen lately) everything enqueued on the step stream so far
    lamb1b_ctx::Staging* e = nullptr;
    for (lamb1b_ctx::Staging& s : ctx->stg)
        if (s.ptr == staging) e = &s;
    bool known = e != nullptr;
    if (!known) {
        e = &ctx->stg[0];
        for (lamb1b_ctx::Staging& s : ctx->stg)
            if (s.last < e->last) e = &s;
        e->ptr = staging;
        e->recorded = false;
    }
    if ((rc = make_event(&e->used))) return rc;
    e->last = ++ctx->stg_clock;

    NvtxRange range("lamb1b compression step from host gradients");
    const int64_t es = host_grads->kind == LAMB1B_GRAD_F32 ? 4 : 2;
    const size_t bytes = (size_t)ctx->P.W * (size_t)host_grads->ld * (size_t)es;
    bool ok = true;
    if (known && e->recorded) {
        ok = cudaStreamWaitEvent(cst, e->used, 0) == cudaSuccess;
    } else {
        ok = cudaEventRecord(ctx->fence, st) == cudaSuccess && cudaStreamWaitEvent(cst, ctx->fence, 0) == cudaSuccess;
    }
    ok = ok && cudaMemcpyAsync(staging, host_grads->ptr, bytes, cudaMemcpyHostToDevice, cst) == cudaSuccess &&
         cudaEventRecord(ctx->copied, cst) == cudaSuccess && cudaStreamWaitEvent(st, ctx->copied, 0) == cudaSuccess;
    if (!ok) {
        cudaGetLastError();
        return LAMB1B_ERR_CUDA;
    }
    if ((rc = compress_enqueue(ctx, &dev, st))) return rc;
    ok = cudaEventRecord(e->used, st) == cudaSuccess;
    e->recorded = ok;
    const int64_t nw = (ctx->P.N + 31) / 32;
    if (ok && words_host)
        ok = cudaMemcpyAsync(words_host, ctx->D.signs_s, (size_t)nw * 4, cudaMemcpyDeviceToHost, st) == cudaSuccess;
    if (ok && scales_host)
        ok = cudaMemcpyAsync(scales_host, ctx->D.scale_s, (size_t)ctx->P.K * 4, cudaMemcpyDeviceToHost, st) ==
             cudaSuccess;
    if (!ok) {
        cudaGetLastError();
        return LAMB1B_ERR_CUDA;
    }
    return LAMB1B_OK;
}

extern "C" int lamb1b_state_view(const lamb1b_ctx* ctx, lamb1b_state* out)
{
    if (!ctx || !out) return LAMB1B_ERR_ARG;
    std::memset(out, 0, sizeof(*out));
    const Dev& D = ctx->D;
    out->m = D.m; out->v = D.v; out->v_fresh = D.v_fresh; out->e_w = D.e_w; out->e_s = D.e_s;
    out->signs_w = D.signs_w; out->signs_s = D.signs_s;
    out->scale_w = D.scale_w; out->scale_s = D.scale_s;
    out->c_bar = D.c_bar; out->r_prev = D.r_prev; out->c_cur = D.c_cur; out->R_last = D.R_last;
    out->Sx = D.Sx; out->Su = D.Su;
    out->N = ctx->P.N; out->Np = ctx->P.Np; out->K = ctx->P.K; out->words_ld = ctx->P.words_ld;
    out->L = ctx->P.L; out->W = ctx->P.W; out->C = ctx->P.C;
    out->stage = ctx->stage; out->t = ctx->t; out->n_warmup = ctx->n_warm;
    return LAMB1B_OK;
}

extern "C" int lamb1b_set_counters(lamb1b_ctx* ctx, int64_t t, int32_t n_warmup, int32_t stage)
{
    if (!ctx) return LAMB1B_ERR_ARG;
    if (t < 0 || t > 0xFFFFFFFFll || n_warmup < 0 || n_warmup > t || (stage != 0 && stage != 1))
        return LAMB1B_ERR_ARG;
    ctx->t = t;
    ctx->n_warm = n_warmup;
    ctx->stage = stage;
    ctx->d_frz_valid = false;    // v may have been rewritten: rebuilt before the next step
    return LAMB1B_OK;
}

extern "C" int lamb1b_check_status(lamb1b_ctx* ctx, void* stream)
{
    if (!ctx) return LAMB1B_ERR_ARG;
    int rc = device_check(ctx);
    if (rc) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint32_t flags = 0;
    if (cudaMemcpyAsync(&flags, ctx->D.flags, sizeof(flags), cudaMemcpyDeviceToHost, st) != cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess)
        return LAMB1B_ERR_CUDA;
    if (flags & 3u) {
        if (cudaMemsetAsync(ctx->D.flags, 0, sizeof(uint32_t), st) != cudaSuccess ||
            cudaStreamSynchronize(st) != cudaSuccess)
            return LAMB1B_ERR_CUDA;
        return (flags & 2u) ? LAMB1B_ERR_TIMEOUT : LAMB1B_ERR_NONFINITE;
    }
    return LAMB1B_OK;
}

extern "C" int lamb1b_set_trace_events(lamb1b_ctx* ctx, void* const* events, int32_t n)
{
    if (!ctx) return LAMB1B_ERR_ARG;
    if (n == 0) {
        ctx->tracing = false;
        return LAMB1B_OK;
    }
    if (n != 4 || !events) return LAMB1B_ERR_ARG;
    for (int i = 0; i < 4; ++i) {
        if (!events[i]) return LAMB1B_ERR_ARG;
    }
    for (int i = 0; i < 4; ++i) ctx->ev[i] = static_cast<cudaEvent_t>(events[i]);
    ctx->tracing = true;
    return LAMB1B_OK;
}

extern "C" int lamb1b_sync_momentum(lamb1b_ctx* ctx, void* stream)
{
    if (!ctx) return LAMB1B_ERR_ARG;
    if (!(ctx->stage == 1 && ctx->t > ctx->n_warm)) return LAMB1B_OK;   // m is dense
    int rc = device_check(ctx);
    if (rc) return rc;
    NvtxRange range("lamb1b sync momentum");
    if (lamb1b::launch_unpack_momentum(ctx->P, ctx->D, static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return LAMB1B_ERR_CUDA;
    return LAMB1B_OK;
}

extern "C" int lamb1b_set_fault_injection(lamb1b_ctx* ctx, int32_t skip_copy, uint32_t wait_tries)
{
    if (!ctx || skip_copy < -1) return LAMB1B_ERR_ARG;
    ctx->P.skip_copy = skip_copy;
    ctx->P.wait_tries = wait_tries ? wait_tries : lamb1b::kDefaultWaitTries;
    return LAMB1B_OK;
}

extern "C" int lamb1b_destroy(lamb1b_ctx* ctx)
{
    delete ctx;
    return LAMB1B_OK;
}

extern "C" const char* lamb1b_error_string(int code)
{
    switch (code) {
    case LAMB1B_OK: return "ok";
    case LAMB1B_ERR_ARG: return "invalid argument";
    case LAMB1B_ERR_ALIGN: return "misaligned pointer or leading dimension";
    case LAMB1B_ERR_WORKSPACE: return "workspace too small";
    case LAMB1B_ERR_STATE: return "call out of order (init, warmup*, freeze, compress*)";
    case LAMB1B_ERR_CUDA: return "CUDA runtime error";
    case LAMB1B_ERR_NONFINITE: return "non-finite gradient seen";
    case LAMB1B_ERR_DEVICE: return "current device is not the context's device";
    case LAMB1B_ERR_TIMEOUT: return "a kernel gave up waiting for its bulk copies";
    default: return "unknown error";
    }
}
