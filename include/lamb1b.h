/*
 * lamb1b: the data-parallel hot path of 1-bit LAMB on one GPU (C ABI).
 *
 * Method: "1-bit LAMB: Communication Efficient Large-Scale Large-Batch
 * Training with LAMB's Convergence Speed" (Li, Awan, Tang, Rajbhandari, He;
 * arXiv 2104.06069).  Citations below name a section of that paper's HTML
 * text ("1-bit LAMB, <section>"); its headings were lost in extraction, so
 * sections are named by their content.  Two stages over a flat binary32
 * parameter buffer cut into per-tensor "layers":
 *   - warmup: LAMB (Adam moments plus one clipped trust ratio per tensor;
 *     1-bit LAMB, background section on LAMB, with its footnote 4 for the
 *     clip definition);
 *   - compression: for W data-parallel workers held side by side in device
 *     memory, error-compensated 1-bit compression of each worker's momentum
 *     (one scale per chunk plus sign bits packed 32 per word; 1-bit LAMB,
 *     background section on error-compensated compression), the compressed
 *     allreduce's gather, average and scatter phases (1-bit LAMB, section 5,
 *     the NCCL-based backend) with server-side error feedback, and the
 *     frozen-variance update with the layerwise factor computed from the
 *     reconstructed gradient under soft thresholds (1-bit LAMB, section 4
 *     summary of the algorithm).
 *
 * Conventions shared by every entry point:
 *   - Pointers named *_dev are device pointers on the device that was current
 *     when lamb1b_init ran; that device must be current for every later call
 *     on the context (LAMB1B_ERR_DEVICE otherwise).
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Every call only enqueues work on it and returns; nothing
 *     synchronises the host except lamb1b_check_status.
 *   - The caller owns all device memory: parameters, gradients and the
 *     workspace.  The library never allocates device memory; it owns only
 *     the host-side context.
 *   - Every call returns 0 or a negative LAMB1B_ERR_* code; nothing aborts
 *     and no kernel traps.  A failed argument check changes no state.
 *   - A context is not thread-safe; calls on one context must not overlap.
 *
 * Arithmetic is binary32 with one rounding per operation in a fixed order
 * (no contraction into fused multiply-add); every sum of squares follows the
 * canonical pairwise tree: one pairwise tree per aligned 256-element granule
 * of the flat buffer (leaves outside the summed segment are +0), then one
 * pairwise tree over the segment's granule sums in order.
 */
#ifndef LAMB1B_H
#define LAMB1B_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum {
    LAMB1B_OK = 0,
    LAMB1B_ERR_ARG = -1,        /* bad size, table, hyper-parameter or NULL     */
    LAMB1B_ERR_ALIGN = -2,      /* pointer or leading dimension misaligned      */
    LAMB1B_ERR_WORKSPACE = -3,  /* workspace smaller than lamb1b_workspace_bytes */
    LAMB1B_ERR_STATE = -4,      /* call out of order: init, warmup*, freeze, compress* */
    LAMB1B_ERR_CUDA = -5,       /* a CUDA runtime call or launch failed         */
    LAMB1B_ERR_NONFINITE = -6,  /* check_finite saw a NaN/Inf gradient          */
    LAMB1B_ERR_DEVICE = -7,     /* current device differs from the context's    */
    LAMB1B_ERR_TIMEOUT = -8     /* a kernel gave up waiting for its own bulk copies
                                   (bounded wait; never expected); the step's
                                   results are not valid                        */
};

/* One tensor of the model (1-bit LAMB, background section on LAMB: every
 * tensor, weight or bias, has its own scaling coefficient).  Tensors are contiguous and ascending:
 * layer[0].offset == 0, layer[l+1].offset == layer[l].offset + layer[l].numel,
 * numel >= 1; N = sum of numel. */
typedef struct {
    int64_t offset;
    int64_t numel;
} lamb1b_layer;

typedef struct {
    int32_t W;                /* virtual data-parallel workers, 1..256          */
    int32_t chunk;            /* C: elements per compression chunk, a power of
                                 two in [256, 8192]; chunk k = [kC, min(kC+C,N)) */
    float lr;                 /* gamma                                          */
    float beta1, beta2;       /* moment decay factors                           */
    float eps;                /* eta, added to sqrt(v)                          */
    float weight_decay;       /* lambda, decoupled, inside the update direction */
    float coeff_min, coeff_max; /* clip bounds of the warmup trust ratio        */
    float coeff_ema;          /* c_bar = ema*c_bar + (1-ema)*c over warmup       */
    float factor_min, factor_max; /* hard bounds of the compression-stage factor */
    float factor_threshold;   /* soft threshold: factor moves at most this
                                 fraction of its previous value per step         */
    int32_t check_finite;     /* 1: flag NaN/Inf gradients (lamb1b_check_status) */
    int32_t variant;          /* 0: 1-bit LAMB.  1: 1-bit Adam (the predecessor
                                 method in the 1-bit LAMB background): Adam in the
                                 warmup, the same compressed momentum exchange in
                                 the compression stage, no layerwise coefficient
                                 (c = 1), no fresh variance; coeff_* and factor_*
                                 are then unused. */
    int32_t error_storage;    /* element type of the worker and server error
                                 buffers (e_w, e_s): 0 binary32; 1 bfloat16,
                                 rounded to nearest even when stored (NaN is
                                 stored as 0x7FC0) and widened exactly when
                                 read.  A storage variant with no counterpart in
                                 the paper: it halves the largest per-worker
                                 traffic at the cost of rounding the kept
                                 compression error to 8 significant bits. */
} lamb1b_hparams;

typedef enum {
    LAMB1B_GRAD_F32 = 0,      /* binary32 [W][ld] in device memory              */
    LAMB1B_GRAD_BF16 = 1,     /* bfloat16 bit patterns [W][ld] in device memory */
    LAMB1B_GRAD_PHILOX = 2    /* generated inside the kernels (see below)       */
} lamb1b_grad_kind;

/* Gradients of one step for all W workers.
 *   F32 / BF16: ptr is a device array of W rows; row w (worker w) starts at
 *     element w*ld; ld >= N and ld*element_size is a multiple of 16 bytes; the
 *     allocation covers W*ld elements; ptr is 16-byte aligned.  Read only.
 *   PHILOX: nothing is read from ptr; element i of worker w at global step t
 *     is drawn from Philox4x32-10 keyed by `seed` (the synthetic-workload
 *     definition of include/lamb1b_gen.h): layer_std[l] * N(0,1) for tensor l,
 *     or heavy_scale * Student-t(3) where layer_heavy[l] != 0.  layer_std and
 *     layer_heavy are device arrays of L entries.
 * A step returns LAMB1B_ERR_ARG, before any launch, when ptr (F32 / BF16) or
 * layer_std / layer_heavy (PHILOX) is not memory of the context's GPU. */
typedef struct {
    int32_t kind;
    int32_t pad0;
    const void* ptr;
    int64_t ld;
    uint64_t seed;
    const float* layer_std;
    const uint8_t* layer_heavy;
    float heavy_scale;
    int32_t pad1;
} lamb1b_grads;

/* Device views of the optimizer state inside the workspace (for inspection,
 * checkpointing and restore; the caller may read or overwrite them between
 * calls).  The momentum: after a compression step m is exactly the server's
 * sign times its chunk scale, and the library keeps it in that form only
 * (signs_s, scale_s, 1/32 of the bytes): the dense m is current in the warmup
 * stage and right after the freeze, and after a compression step only once
 * lamb1b_sync_momentum has written it.  From the first compression step on,
 * signs_s and scale_s are the momentum a later step reads; a restore must
 * write them (the counters passed to lamb1b_set_counters tell the library
 * which form is current: t > n_warmup in the compression stage).  Likewise v
 * is frozen in the compression stage and the library keeps fl(sqrt(v) + eps)
 * precomputed from it; after rewriting v, call lamb1b_set_counters (as every
 * restore does) and the next step rebuilds it.  Padded layouts: Np = N rounded up to a multiple of max(C, 4096)
 * elements per vector (>= K*C), words_ld = Np/32.
 *   m, v, v_fresh: [Np] binary32; elements >= N are kept at 0
 *   e_s: [Np], e_w: [W][Np], binary32 or (error_storage = 1) bfloat16 bits
 *   signs_w: [W][words_ld] u32;   signs_s: [words_ld]
 *   scale_w: [W][K];   scale_s: [K]
 *   c_bar, r_prev, c_cur, R_last, Sx, Su: [L]
 * Sign words: element j at word j/32, bit j%32, bit = 1 for a +1 sign. */
typedef struct {
    float* m;
    float* v;
    float* v_fresh;
    void* e_w;          /* element type per lamb1b_hparams.error_storage    */
    void* e_s;
    uint32_t* signs_w;
    uint32_t* signs_s;
    float* scale_w;
    float* scale_s;
    float* c_bar;       /* average of the warmup coefficients               */
    float* r_prev;      /* compression-stage factor of the last step        */
    float* c_cur;       /* coefficient applied by the last step             */
    float* R_last;      /* last step's per-tensor max ratio                 */
    float* Sx;          /* last warmup step's per-tensor sum of x^2         */
    float* Su;          /* last warmup step's per-tensor sum of u^2         */
    int64_t N, Np, K, words_ld;
    int32_t L, W, C;
    int32_t stage;      /* 0 warmup, 1 compression                          */
    int64_t t;          /* steps taken (global step counter)                */
    int32_t n_warmup;   /* warmup steps taken                               */
    int32_t pad0;
} lamb1b_state;

/* Bytes of device workspace lamb1b_init needs for this table and settings;
 * 0 when the arguments are invalid.  Pure host function. */
size_t lamb1b_workspace_bytes(const lamb1b_layer* layers, int32_t L,
                              const lamb1b_hparams* hp);

/* Opaque host-side context. */
typedef struct lamb1b_ctx lamb1b_ctx;

/* Validates the table and settings, lays out the caller's workspace
 * (workspace_dev 256-byte aligned, at least lamb1b_workspace_bytes bytes),
 * uploads the tables and zeroes the state (m = v = 0, c_bar = r_prev = c_cur
 * = 1) on `stream`.  params_dev (N binary32, 16-byte aligned) is updated in
 * place by every step.  `layers` is copied; the caller may free it.  On
 * success *out receives a context that lamb1b_destroy frees.
 * Errors: ARG (table, sizes, settings, NULL), ALIGN, WORKSPACE, CUDA. */
int lamb1b_init(lamb1b_ctx** out, const lamb1b_layer* layers, int32_t L,
                const lamb1b_hparams* hp, float* params_dev,
                void* workspace_dev, size_t workspace_bytes, void* stream);

/* Warmup stage, one LAMB step (1-bit LAMB, background section on LAMB: the
 * symbol list and clip definition of its update rule; the introduction: LAMB
 * runs uncompressed as the warmup stage):
 *   gbar = (sum_w g_w) / W, summed in ascending w
 *   m = beta1 m + (1-beta1) gbar;  v = beta2 v + (1-beta2) gbar^2
 *   u = m / (sqrt(v) + eps) + weight_decay x
 *   c_l = clip(||x_l|| / ||u_l||, coeff_min, coeff_max)  (1 if a norm is 0)
 *   x = x - (lr c_l) u;  c_bar_l = c_l on the first warmup step, then
 *   coeff_ema c_bar_l + (1-coeff_ema) c_l
 * Errors: STATE after lamb1b_freeze_variance; ARG/ALIGN for bad gradients. */
int lamb1b_warmup_step(lamb1b_ctx* ctx, const lamb1b_grads* grads, void* stream);

/* Stage switch (1-bit LAMB, background section on 1-bit Adam, and the
 * 1-bit Adam abstract: the variance is frozen after the warmup): v is kept as
 * the fixed preconditioner, v_fresh = v, worker and server errors = 0,
 * r_prev = 1; c_bar is fixed from here on.  Allowed once, before any
 * compression step.  Errors: STATE. */
int lamb1b_freeze_variance(lamb1b_ctx* ctx, void* stream);

/* Compression stage, one step (1-bit LAMB: the introduction's compression
 * stage, momentum SGD preconditioned by the frozen variance; the background
 * section on error-compensated compression for the worker and server
 * compressors; section 5 for the gather, average and scatter phases; the
 * section 4 summary for the reconstructed gradient and the soft thresholds).
 * Per chunk k and worker w (gather phase):
 *   z = (beta1 m + (1-beta1) g_w) + e_w
 *   s_wk = sqrt(sum_chunk z^2 / n_k);  bit = !(z < 0);  e_w = z -+ s_wk
 * server (average and scatter phases):
 *   a = sum over w ascending of +-s_wk;  y = a / W + e_s
 *   s_k = sqrt(sum_chunk y^2 / n_k);  e_s = y -+ s_k;  m_new = +-s_k
 * reconstructed gradient g~ = (m_new - beta1 m) / (1-beta1),
 *   v_fresh = beta2 v_fresh + (1-beta2) g~^2,
 *   R_l = max over tensor l of (sqrt(v)+eps) / (sqrt(v_fresh)+eps)
 *   r_l = clip(clip(R_l, factor_min, factor_max),
 *              (1-factor_threshold) r_prev_l, (1+factor_threshold) r_prev_l)
 *   c_l = c_bar_l r_l;  m = m_new;  x = x - (lr c_l)(m / (sqrt(v)+eps) + wd x)
 * The packed words and scales of every worker and of the server are left in
 * the workspace (lamb1b_state_view); the new m is kept as the server's words
 * and scales (signs_s, scale_s) and written densely only by
 * lamb1b_sync_momentum.  Enqueues kernels only (no host synchronisation, no
 * allocation), so a step can be captured in a CUDA graph; the host step
 * counter advances on direct calls.  Errors: STATE before the freeze. */
int lamb1b_compress_step(lamb1b_ctx* ctx, const lamb1b_grads* grads, void* stream);

/* The same compression step with its gradients in host memory, for callers
 * whose gradients arrive on the host: the step copies them to the GPU, runs,
 * and reads the server's message back.
 *   host_grads   kind LAMB1B_GRAD_F32 or LAMB1B_GRAD_BF16; ptr = W rows of
 *                ld elements in pinned (page-locked) host memory, the layout
 *                lamb1b_compress_step takes on the device.
 *   staging      a caller-owned device buffer of W x ld elements of the same
 *                type on the context's GPU (16-byte aligned, ld x element
 *                size a multiple of 16 bytes): the copy's destination.
 *   words_host   pinned host memory for the step's server sign words,
 *                ceil(N/32) uint32 (the signs_s of lamb1b_state_view), or NULL.
 *   scales_host  pinned host memory for its K chunk scales (scale_s), or NULL.
 *   stream       the stream of the step's kernels and of the read-back.
 *   copy_stream  the stream of the host-to-device copy (may be `stream`).
 * Order: the copy runs on copy_stream after the work already enqueued there
 * and after the last step of this context that read `staging` (the context
 * remembers the last 4 staging buffers; for any other buffer the copy waits
 * for all work enqueued on `stream` so far, so pass the same `stream` to
 * every step of a context); the kernels wait for the copy; the read-back
 * follows the kernels on `stream`.  So with two staging buffers used in turn
 * and a separate copy_stream, a step's copy overlaps the previous step's
 * kernels.  The host buffers must stay valid and unchanged until `stream`
 * has passed the step.  Not for stream capture: on a capturing stream it
 * returns LAMB1B_ERR_ARG and enqueues nothing.
 * Errors: STATE before the freeze; ARG (other gradient kinds, pageable or
 * device memory where pinned host memory is required, staging not memory of
 * the context's GPU, ld < N, a capturing stream); ALIGN; CUDA. */
int lamb1b_compress_step_host(lamb1b_ctx* ctx, const lamb1b_grads* host_grads, void* staging,
                              uint32_t* words_host, float* scales_host, void* stream,
                              void* copy_stream);

/* Fills *out with device pointers into the workspace and the counters. */
int lamb1b_state_view(const lamb1b_ctx* ctx, lamb1b_state* out);

/* Restores the counters after the caller has written a saved state into the
 * workspace through lamb1b_state_view (checkpoint resume).  stage 0 or 1. */
int lamb1b_set_counters(lamb1b_ctx* ctx, int64_t t, int32_t n_warmup, int32_t stage);

/* Synchronises `stream` and reports (then clears) the device status flags
 * raised since the last check: LAMB1B_ERR_TIMEOUT if a compression kernel gave
 * up waiting for its own shared-memory bulk copies, else LAMB1B_ERR_NONFINITE
 * if a step run with check_finite = 1 saw a NaN or Inf gradient, else 0. */
int lamb1b_check_status(lamb1b_ctx* ctx, void* stream);

/* Tracing: with n == 4, every later warmup or compression step records
 * events[0] before its first kernel, events[1] after the element-streaming
 * kernel (warmup moments, or the fused worker+server compression), events[2]
 * after the per-tensor kernel and events[3] after the parameter update, all
 * on the step's stream.  events are cudaEvent_t handles owned by the caller
 * and must stay valid while tracing is on.  n == 0 turns tracing off.
 * Errors: ARG for other n or NULL events with n == 4. */
int lamb1b_set_trace_events(lamb1b_ctx* ctx, void* const* events, int32_t n);

/* Writes the dense momentum m (lamb1b_state.m) from the server sign words and
 * chunk scales of the last compression step, on `stream`; a no-op while the
 * dense m is current (warmup stage, and the compression stage before its
 * first step).  Elements >= N stay 0.
 * Errors: ARG for a NULL ctx; DEVICE, CUDA as for the steps. */
int lamb1b_sync_momentum(lamb1b_ctx* ctx, void* stream);

/* Testing hook for the failure path of the compression step (the paper has
 * no counterpart).  The compression kernel stages its inputs through shared
 * memory with bulk copies and waits for each with a bounded mbarrier wait.
 * skip_copy >= 0 makes the first CTA of every later compression step leave
 * out the copy at that position of its copy sequence (0 = the first tile's
 * momentum, then per worker its gradient and error, ...), so the wait for it
 * can only run out; skip_copy = -1 turns this off.  wait_tries bounds the
 * copy waits of that first CTA, in mbarrier.try_wait calls; 0 restores the
 * default (2^24, seconds).  Every other CTA's waits, and the wait with which a
 * CTA that gave up lets its issued copies land before it exits, keep the
 * default bound.  A step whose wait ran out stops early, records LAMB1B_ERR_TIMEOUT for
 * lamb1b_check_status and leaves the optimizer state undefined (restore it
 * from a checkpoint); the CUDA context stays usable.  No GPU fault is raised.
 * Errors: ARG for a NULL ctx or skip_copy < -1. */
int lamb1b_set_fault_injection(lamb1b_ctx* ctx, int32_t skip_copy, uint32_t wait_tries);

/* Allocation-free per-tensor sums of squares (the paper has no counterpart;
 * this is a convenience for callers that cannot allocate device memory).
 *
 * out_dev[l] = sum over tensor l of x_i^2, in the same canonical pairwise-tree
 * order as the warmup step's Sx (lamb1b_state.Sx), for the table `layers`
 * (host array of L entries, contiguous from 0, as for lamb1b_init).
 *
 * Who needs it: code that may not call cudaMalloc/cudaFree or size a
 * workspace -- a plug-in living inside a framework whose caching allocator
 * owns all device memory, or a latency-critical loop where cudaMalloc and
 * cudaFree would synchronise the device.  Such a caller still owns x_dev (N
 * binary32, 16-byte aligned) and out_dev (L binary32); all scratch comes from
 * a fixed array inside this library (about 16 MiB, set aside on every GPU that
 * loads the library until the process exits).  No call allocates.
 *
 * Limits: L <= 4096 and at most 2^22 half-granule partial sums (2 per aligned
 * 256-element granule a tensor meets, so N up to about 5.3e8); larger inputs
 * return LAMB1B_ERR_ARG without touching the GPU.
 * The first call on a device looks up the scratch array's device address for
 * that device; later calls reuse it.  The call stages its tables from host
 * memory that lives only for the call, so it cannot be captured into a CUDA
 * graph: on a stream that is capturing it returns LAMB1B_ERR_ARG and enqueues
 * nothing.  Every call reuses the same scratch, which keeps the previous
 * call's contents; the call clears what it needs.  Calls that overlap on the
 * GPU (different streams, or different host threads) race on the scratch:
 * serialise them.  The host table is staged before the call returns.
 * Errors: ARG, ALIGN (x_dev), CUDA. */
int lamb1b_tensor_sumsq_noalloc(const float* x_dev, const lamb1b_layer* layers, int32_t L,
                                float* out_dev, void* stream);

/* Frees the host context (not the caller's device memory).  NULL is a no-op. */
int lamb1b_destroy(lamb1b_ctx* ctx);

/* Static description of an error code. */
const char* lamb1b_error_string(int code);

#ifdef __cplusplus
}
#endif
#endif
