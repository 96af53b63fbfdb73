/*
 * 1-bit LAMB, data-parallel hot path: plain single-threaded CPU oracle.
 *
 * TEST INFRASTRUCTURE.  This file is the slow, obviously-correct statement of
 * what the GPU library computes.  Only the test suite, the package smoke check
 * and the benchmark's CPU-baseline leg may load it.  It shares no code with the
 * GPU library.
 *
 * Sources (1-bit LAMB, Li et al., arXiv 2104.06069, HTML text):
 *   - introduction: the method has two stages, LAMB as warmup, then momentum
 *     SGD with 1-bit compressed communication "pre-conditioned" by the warmup
 *     state, with layerwise learning rates adapted from both stages;
 *   - background, "error-compensated compression": compress the input plus
 *     the previous step's compression error and keep the new error; 1-bit
 *     compression sends +-1 signs and a scale;
 *   - background, "1-bit Adam": the variance is frozen after warmup and used
 *     as a fixed preconditioner; the momentum is what gets compressed;
 *   - background, "LAMB": Adam moments plus one scaling coefficient per tensor
 *     (weight and bias each have their own), clip applied to the whole ratio,
 *     clip(x, a, b) = min{max{x, a}, b} (footnote 4);
 *   - section 4 summary: in the compression stage the layerwise rate is
 *     updated from a "reconstructed gradient" built from the compressed
 *     momentum, with extra "stabilized soft thresholds";
 *   - section 5 summary: compressed allreduce in three phases: gather (worker
 *     i receives chunk i from everybody), average, scatter.
 *
 * The LAMB update display and the 1-bit LAMB algorithm listing are not in the
 * extracted text; where the text is silent this file takes these readings:
 *   u = m / (sqrt(v) + eps) + wd * x, no bias correction; c = clip(||x||/||u||,
 *   cmin, cmax), 1 when either norm is 0; warmup gradient = plain mean of the
 *   W workers' gradients; chunk scale = ||z||_2 / sqrt(n_k); sign bit = !(z < 0),
 *   LSB first, 32 elements per word; server average = sum over workers in
 *   ascending order of +-scale, divided by W; every worker's momentum becomes
 *   the decompressed server result; reconstructed gradient
 *   g~ = (m_new - beta1 m_old) / (1 - beta1); a fresh second moment v_f is
 *   tracked from g~; per tensor R = max (sqrt(v_frozen)+eps)/(sqrt(v_f)+eps);
 *   soft thresholds: r = clip(clip(R, fmin, fmax), (1-thr) r_prev,
 *   (1+thr) r_prev), c = c_bar * r with c_bar the exponential moving average of
 *   the warmup coefficients.  Variant 1 is 1-bit Adam (the 1-bit Adam page and
 *   the 1-bit LAMB background on it): vanilla Adam in the warmup, the same
 *   compressed momentum exchange in the compression stage, no layerwise
 *   coefficient and no fresh variance.  err_bf16 = 1 stores the worker and
 *   server errors rounded to bfloat16 (a storage variant, not in the paper).
 *   Parity with the published algorithm is unpinned
 *   for those readings (bias correction, clip bounds, scale formula, c_bar,
 *   fresh variance, soft thresholds); the pins here are the stated invariants.
 *
 * Arithmetic: binary32, every operation rounded once (build with
 * -ffp-contract=off, no fast-math).  Sums of squares follow one fixed
 * association, the canonical pairwise tree (cpt_sumsq below), so that the
 * result is a function of the inputs alone.
 */
#include <float.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    /* problem */
    int64_t N;
    int32_t L, W, C;
    int32_t variant;        /* 0: 1-bit LAMB, 1: 1-bit Adam (no layerwise scaling) */
    const int64_t* off;     /* [L] first flat index of tensor l   */
    const int64_t* numel;   /* [L] element count of tensor l      */
    /* hyper-parameters */
    float lr, beta1, beta2, eps, wd;
    float cmin, cmax, cema;
    float fmin, fmax, fthr;
    int32_t err_bf16;       /* 1: worker and server errors are stored as bf16 */
    /* state, caller-owned */
    float* x;               /* [N] parameters                      */
    float* m;               /* [N] momentum                        */
    float* v;               /* [N] second moment (frozen later)    */
    float* v_fresh;         /* [N] second moment of g~             */
    float* e_w;             /* [W][N] worker compression errors    */
    float* e_s;             /* [N] server compression error        */
    uint32_t* signs_w;      /* [W][NW] worker sign words           */
    uint32_t* signs_s;      /* [NW] server sign words              */
    float* scale_w;         /* [W][K] worker chunk scales          */
    float* scale_s;         /* [K] server chunk scales             */
    float* c_bar;           /* [L] warmup coefficient average      */
    float* r_prev;          /* [L] last compression-stage factor   */
    float* c_cur;           /* [L] coefficient used by the last step */
    float* R;               /* [L] last per-tensor max ratio       */
    float* Sx;              /* [L] last warmup sum of x^2          */
    float* Su;              /* [L] last warmup sum of u^2          */
    int64_t t;              /* steps taken                         */
    int32_t n_warm;         /* warmup steps taken                  */
    int32_t stage;          /* 0 warmup, 1 compression             */
} orc_t;

/* ---- one-rounding helpers (names make the rounding points explicit) ----
 * Each returns the binary32 result of one IEEE operation.  This relies on
 * FLT_EVAL_METHOD == 0 (checked below) and on -ffp-contract=off, so that no
 * product is fused into a following sum. */
#if !defined(FLT_EVAL_METHOD) || FLT_EVAL_METHOD != 0
#error "the oracle needs binary32 expression evaluation (FLT_EVAL_METHOD == 0)"
#endif
static float fadd(float a, float b) { return a + b; }
static float fsub(float a, float b) { return a - b; }
static float fmul(float a, float b) { return a * b; }
static float fdiv(float a, float b) { return a / b; }
static float fsqrt(float a) { return sqrtf(a); }
/* clip(x, a, b) = min{max{x, a}, b} written with comparisons (NaN passes) */
static float clip(float x, float a, float b)
{
    float r = (x < a) ? a : x;
    return (r > b) ? b : r;
}

/* Round a binary32 value to the nearest bfloat16 (ties to even) and widen it
 * back; NaN becomes the quiet NaN 0x7FC0.  Storage rounding of the
 * error-feedback buffers in the bf16 error-storage variant. */
float orc_bf16_round(float x)
{
    uint32_t b;
    memcpy(&b, &x, 4);
    uint32_t h = (x != x) ? 0x7FC0u : ((b + 0x7FFFu + ((b >> 16) & 1u)) >> 16);
    uint32_t r = h << 16;
    float y;
    memcpy(&y, &r, 4);
    return y;
}

/* the error buffers keep exactly what the storage format can hold */
static float store_err(const orc_t* s, float e) { return s->err_bf16 ? orc_bf16_round(e) : e; }

/* ---- canonical pairwise tree ------------------------------------------ */

/* T(v[0..n)) for n a power of two: T(v) = T(left half) + T(right half). */
static float tree(const float* v, int64_t n)
{
    if (n == 1) return v[0];
    float a = tree(v, n / 2);
    float b = tree(v + n / 2, n / 2);
    return fadd(a, b);
}

static int64_t next_pow2(int64_t n)
{
    int64_t p = 1;
    while (p < n) p <<= 1;
    return p;
}

/*
 * Sum of squares over the flat-index segment [lo, hi).  Element i's value is
 * a[i - a0].  Leaves are fl(a_i * a_i) inside the segment and +0 outside.
 * Level 0: one tree per aligned 256-element granule that meets the segment.
 * Level 1: one tree over those granule sums in granule order, zero-padded to
 * a power of two.
 */
float orc_cpt_sumsq(const float* a, int64_t a0, int64_t lo, int64_t hi)
{
    if (hi <= lo) return 0.0f;
    int64_t g0 = lo / 256, g1 = (hi - 1) / 256;
    int64_t ng = g1 - g0 + 1, np2 = next_pow2(ng);
    float* part = (float*)calloc((size_t)np2, sizeof(float));
    float leaf[256];
    for (int64_t g = g0; g <= g1; ++g) {
        for (int j = 0; j < 256; ++j) {
            int64_t i = g * 256 + j;
            leaf[j] = (i >= lo && i < hi) ? fmul(a[i - a0], a[i - a0]) : 0.0f;
        }
        part[g - g0] = tree(leaf, 256);
    }
    float s = tree(part, np2);
    free(part);
    return s;
}

/* ---- 1-bit compressor (error-compensated, one scale per chunk) --------- */

/*
 * Compress z (n values of a chunk that starts at flat index k*C; slots past
 * n are padding) into one scale and sign bits, and produce the new error.
 *   scale = sqrt(S / n), S = canonical sum of z^2 over the chunk
 *   bit   = !(z < 0)    (so +0, -0 and NaN send +1), 0 for padding
 *   err   = z - sigma * scale
 * words receives C/32 words, element j of the chunk at word j/32 bit j%32.
 */
static float compress_chunk(const float* z, int64_t k, int32_t C, int64_t n,
                            uint32_t* words, float* err)
{
    float S = orc_cpt_sumsq(z, k * (int64_t)C, k * (int64_t)C, k * (int64_t)C + n);
    float s = fsqrt(fdiv(S, (float)n));
    for (int32_t q = 0; q < C / 32; ++q) words[q] = 0u;
    for (int64_t j = 0; j < n; ++j) {
        int pos = !(z[j] < 0.0f);
        if (pos) words[j / 32] |= 1u << (j % 32);
        err[j] = pos ? fsub(z[j], s) : fadd(z[j], s);
    }
    return s;
}

/* exported for pin tests: compress one chunk in isolation */
float orc_compress_chunk(const float* z, int64_t k, int32_t C, int64_t n,
                         uint32_t* words, float* err)
{
    return compress_chunk(z, k, C, n, words, err);
}

/* ---- warmup stage: LAMB --------------------------------------------------- */

/*
 * One LAMB step on the mean of the W workers' gradients g[w*ld + i].
 *   gbar = (sum_w g_w) / W                     (uncompressed averaging)
 *   m = b1 m + (1-b1) gbar ; v = b2 v + (1-b2) gbar^2
 *   u = m / (sqrt(v) + eps) + wd x
 *   c_l = clip(||x_l|| / ||u_l||, cmin, cmax)  (1 if a norm is 0)
 *   x = x - (lr c_l) u
 * c_bar_l: first warmup step c_l, then c_bar = cema c_bar + (1-cema) c_l.
 */
int orc_warmup_step(orc_t* s, const float* g, int64_t ld)
{
    if (s->stage != 0) return -4;
    const int64_t N = s->N;
    const float w1 = fsub(1.0f, s->beta1), w2 = fsub(1.0f, s->beta2);
    float* u = (float*)malloc((size_t)N * sizeof(float));
    for (int64_t i = 0; i < N; ++i) {
        float acc = 0.0f;
        for (int32_t w = 0; w < s->W; ++w) acc = fadd(acc, g[(int64_t)w * ld + i]);
        float gb = fdiv(acc, (float)s->W);
        s->m[i] = fadd(fmul(s->beta1, s->m[i]), fmul(w1, gb));
        s->v[i] = fadd(fmul(s->beta2, s->v[i]), fmul(w2, fmul(gb, gb)));
        float d = fadd(fsqrt(s->v[i]), s->eps);
        u[i] = fadd(fdiv(s->m[i], d), fmul(s->wd, s->x[i]));
    }
    const float one_m_ema = fsub(1.0f, s->cema);
    for (int32_t l = 0; l < s->L; ++l) {
        int64_t lo = s->off[l], hi = lo + s->numel[l];
        if (s->variant == 1) {
            /* 1-bit Adam's warmup is vanilla Adam: no layerwise coefficient */
            float gl = s->lr;
            for (int64_t i = lo; i < hi; ++i) s->x[i] = fsub(s->x[i], fmul(gl, u[i]));
            continue;
        }
        float sx = orc_cpt_sumsq(s->x, 0, lo, hi);
        float su = orc_cpt_sumsq(u, 0, lo, hi);
        float ratio = (sx == 0.0f || su == 0.0f) ? 1.0f : fdiv(fsqrt(sx), fsqrt(su));
        float c = clip(ratio, s->cmin, s->cmax);
        s->Sx[l] = sx;
        s->Su[l] = su;
        s->c_cur[l] = c;
        s->c_bar[l] = (s->n_warm == 0) ? c
                      : fadd(fmul(s->cema, s->c_bar[l]), fmul(one_m_ema, c));
        float gc = fmul(s->lr, c);
        for (int64_t i = lo; i < hi; ++i) s->x[i] = fsub(s->x[i], fmul(gc, u[i]));
    }
    free(u);
    s->n_warm += 1;
    s->t += 1;
    return 0;
}

/* ---- stage switch: freeze the second moment ------------------------------ */
int orc_freeze(orc_t* s)
{
    if (s->stage != 0) return -4;
    const int64_t N = s->N;
    memcpy(s->v_fresh, s->v, (size_t)N * sizeof(float));
    memset(s->e_w, 0, (size_t)s->W * (size_t)N * sizeof(float));
    memset(s->e_s, 0, (size_t)N * sizeof(float));
    for (int32_t l = 0; l < s->L; ++l) { s->r_prev[l] = 1.0f; s->R[l] = 0.0f; }
    s->stage = 1;
    return 0;
}

/* ---- compression stage ------------------------------------------------ */

/*
 * Chunk k of one compression step: every worker's error-compensated 1-bit
 * compression of its momentum, then the server's average, recompression and
 * scatter, then the reconstructed gradient and the fresh second moment.
 * rho[j] receives (sqrt(v)+eps)/(sqrt(v_f)+eps) for chunk element j.
 * Only chunk k's slices of the state are read and written.
 */
int orc_compress_chunk_step(orc_t* s, const float* g, int64_t ld, int64_t k, float* rho)
{
    const int64_t N = s->N, C = s->C;
    const int64_t K = (N + C - 1) / C, NW = (N + 31) / 32;
    if (k < 0 || k >= K) return -1;
    const int64_t base = k * C;
    const int64_t n = (base + C <= N) ? C : N - base;
    const float w1 = fsub(1.0f, s->beta1), w2 = fsub(1.0f, s->beta2);
    float* z = (float*)calloc((size_t)C, sizeof(float));
    float* err = (float*)calloc((size_t)C, sizeof(float));
    float* acc = (float*)calloc((size_t)C, sizeof(float));     /* server sum, starts at +0 */
    uint32_t* words = (uint32_t*)calloc((size_t)C / 32, sizeof(uint32_t));
    const int64_t q0 = base / 32;
    const int64_t nq = (n + 31) / 32;   /* words of this chunk that exist */

    /* phase 1 (gather): each worker compresses its chunk k */
    for (int32_t w = 0; w < s->W; ++w) {
        float* ew = s->e_w + (int64_t)w * N;
        for (int64_t j = 0; j < n; ++j) {
            int64_t i = base + j;
            float mw = fadd(fmul(s->beta1, s->m[i]), fmul(w1, g[(int64_t)w * ld + i]));
            z[j] = fadd(mw, ew[i]);
        }
        float sc = compress_chunk(z, k, (int32_t)C, n, words, err);
        for (int64_t j = 0; j < n; ++j) ew[base + j] = store_err(s, err[j]);
        for (int64_t q = 0; q < nq; ++q) s->signs_w[(int64_t)w * NW + q0 + q] = words[q];
        s->scale_w[(int64_t)w * K + k] = sc;
        /* phase 2 (average), accumulated in worker order */
        for (int64_t j = 0; j < n; ++j) {
            int pos = (words[j / 32] >> (j % 32)) & 1u;
            acc[j] = fadd(acc[j], pos ? sc : -sc);
        }
    }
    /* server: average, add server error, recompress */
    for (int64_t j = 0; j < n; ++j) {
        float avg = fdiv(acc[j], (float)s->W);
        z[j] = fadd(avg, s->e_s[base + j]);
    }
    float ss = compress_chunk(z, k, (int32_t)C, n, words, err);
    for (int64_t j = 0; j < n; ++j) s->e_s[base + j] = store_err(s, err[j]);
    for (int64_t q = 0; q < nq; ++q) s->signs_s[q0 + q] = words[q];
    s->scale_s[k] = ss;
    /* phase 3 (scatter): every worker's momentum becomes the server result;
     * reconstructed gradient and fresh second moment */
    for (int64_t j = 0; j < n; ++j) {
        int64_t i = base + j;
        int pos = (words[j / 32] >> (j % 32)) & 1u;
        float m_new = pos ? ss : -ss;
        if (s->variant == 1) {      /* 1-bit Adam: no fresh variance, no ratio */
            s->m[i] = m_new;
            if (rho) rho[j] = 1.0f;
            continue;
        }
        float gt = fdiv(fsub(m_new, fmul(s->beta1, s->m[i])), w1);
        s->v_fresh[i] = fadd(fmul(s->beta2, s->v_fresh[i]), fmul(w2, fmul(gt, gt)));
        float num = fadd(fsqrt(s->v[i]), s->eps);
        float den = fadd(fsqrt(s->v_fresh[i]), s->eps);
        float r = fdiv(num, den);
        if (rho) rho[j] = (r != r) ? INFINITY : r;
        s->m[i] = m_new;
    }
    free(z); free(err); free(acc); free(words);
    return 0;
}

/* Per-tensor factor from its max ratio R (soft thresholds around r_prev). */
float orc_layer_factor(float R, float r_prev, float fmin, float fmax, float fthr)
{
    float r = clip(R, fmin, fmax);
    float lo = fmul(fsub(1.0f, fthr), r_prev);
    float hi = fmul(fadd(1.0f, fthr), r_prev);
    return clip(r, lo, hi);
}

/* x = x - (lr c_l) (m / (sqrt(v) + eps) + wd x) over tensor l */
static void update_tensor(orc_t* s, int32_t l, float c)
{
    int64_t lo = s->off[l], hi = lo + s->numel[l];
    float gc = fmul(s->lr, c);
    for (int64_t i = lo; i < hi; ++i) {
        float d = fadd(fsqrt(s->v[i]), s->eps);
        float u = fadd(fdiv(s->m[i], d), fmul(s->wd, s->x[i]));
        s->x[i] = fsub(s->x[i], fmul(gc, u));
    }
}

int orc_compress_step(orc_t* s, const float* g, int64_t ld)
{
    if (s->stage != 1) return -4;
    const int64_t N = s->N, C = s->C;
    const int64_t K = (N + C - 1) / C;
    float* rho = (float*)malloc((size_t)K * (size_t)C * sizeof(float));
    for (int64_t k = 0; k < K; ++k)
        orc_compress_chunk_step(s, g, ld, k, rho + k * C);
    for (int32_t l = 0; l < s->L; ++l) {
        int64_t lo = s->off[l], hi = lo + s->numel[l];
        if (s->variant == 1) {      /* 1-bit Adam: coefficient 1, frozen-variance update */
            update_tensor(s, l, 1.0f);
            continue;
        }
        float R = 0.0f;
        for (int64_t i = lo; i < hi; ++i) R = (rho[i] > R) ? rho[i] : R;
        float r = orc_layer_factor(R, s->r_prev[l], s->fmin, s->fmax, s->fthr);
        s->R[l] = R;
        s->r_prev[l] = r;
        s->c_cur[l] = fmul(s->c_bar[l], r);
        update_tensor(s, l, s->c_cur[l]);
    }
    free(rho);
    s->t += 1;
    return 0;
}
