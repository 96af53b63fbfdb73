/*
 * Seeded synthetic-input generator (host side).
 *
 * This module produces the synthetic workloads the optimizer is run on:
 * initial parameters and per-(worker, step, element) gradients.  It holds
 * none of the optimizer's arithmetic.  It serves both the CPU oracle and the
 * GPU library's tests; the GPU library carries its own CUDA implementation
 * of the same definition for on-device generation, and the two are required
 * to agree bit for bit.
 *
 * Definition (every floating-point step is one IEEE binary32 operation with
 * round-to-nearest-even; no fused multiply-add, no library transcendental):
 *
 *   Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as
 *   easy as 1, 2, 3", SC'11): 10 rounds of the 4x32 S-box with multipliers
 *   0xD2511F53 / 0xCD9E8D57 and Weyl key increments 0x9E3779B9 / 0xBB67AE85.
 *   key = (seed lo32, seed hi32).
 *
 *   uniform(u) = (2*(u >> 9) + 1) * 2^-24, in (0, 1), exact in binary32.
 *
 *   Box-Muller (1958): Z0 = R cos(theta), Z1 = R sin(theta) with
 *   R = sqrt(-2 ln U1), theta = 2 pi U2.  ln, cos and sin are evaluated with
 *   the fixed series below (natural-log atanh series after an exact binade
 *   split; Taylor series for sin and cos after an exact quadrant split), so
 *   every implementation that follows this text gets the same bits.
 *
 *   Element i of a normal stream takes output i % 4 of the Philox call with
 *   counter (q lo32, q hi32, t, stream), q = i / 4; outputs (0,1) and (2,3)
 *   are the two Box-Muller pairs.  Gradients: stream = w.  Parameters:
 *   t = 0, stream = 0x7FFFFFFF.
 *
 *   Student-t with 3 degrees of freedom: one Philox call per element, counter
 *   (i lo32, i hi32, t, 0x80000000 | w), four normals Z0..Z3,
 *   T = Z0 / sqrt(((Z1^2 + Z2^2) + Z3^2) / 3).
 *
 *   bf16 storage: round-to-nearest-even of the binary32 bit pattern.
 */
#include <stdint.h>
#include <string.h>

static inline float f32_from_u32(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }
static inline uint32_t u32_from_f32(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }

/* ---- Philox4x32-10 ---------------------------------------------------- */
void wl_philox4x32_10(const uint32_t ctr_in[4], const uint32_t key_in[2], uint32_t out[4])
{
    uint32_t c0 = ctr_in[0], c1 = ctr_in[1], c2 = ctr_in[2], c3 = ctr_in[3];
    uint32_t k0 = key_in[0], k1 = key_in[1];
    for (int r = 0; r < 10; ++r) {
        if (r > 0) { k0 += 0x9E3779B9u; k1 += 0xBB67AE85u; }
        uint64_t p0 = (uint64_t)0xD2511F53u * (uint64_t)c0;
        uint64_t p1 = (uint64_t)0xCD9E8D57u * (uint64_t)c2;
        uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
        uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
        uint32_t n0 = hi1 ^ c1 ^ k0;
        uint32_t n1 = lo1;
        uint32_t n2 = hi0 ^ c3 ^ k1;
        uint32_t n3 = lo0;
        c0 = n0; c1 = n1; c2 = n2; c3 = n3;
    }
    out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* ---- uniform, log, sincos ----------------------------------------------- */
float wl_uniform(uint32_t u)
{
    return (float)(((u >> 9) << 1) | 1u) * 0x1p-24f;
}

/* natural log for a normal positive binary32 input */
float wl_log(float u)
{
    uint32_t b = u32_from_f32(u);
    int e = (int)((b >> 23) & 0xFFu) - 127;
    float f = f32_from_u32((b & 0x7FFFFFu) | 0x3F800000u);  /* [1, 2) */
    if (f > 0x1.6a09e6p+0f) { f = f * 0.5f; e = e + 1; }    /* [~0.707, ~1.414] */
    float s = (f - 1.0f) / (f + 1.0f);
    float s2 = s * s;
    float q = 0x1.745d18p-3f;                 /* 2/11 */
    q = q * s2 + 0x1.c71c72p-3f;              /* 2/9  */
    q = q * s2 + 0x1.24924ap-2f;              /* 2/7  */
    q = q * s2 + 0x1.99999ap-2f;              /* 2/5  */
    q = q * s2 + 0x1.555556p-1f;              /* 2/3  */
    float lnf = (2.0f * s) + (s * s2) * q;
    return (float)e * 0x1.62e430p-1f + lnf;   /* e ln2 + ln f */
}

/* cos and sin of 2*pi*v for v in [0, 1) */
void wl_sincos2pi(float v, float* c_out, float* s_out)
{
    float q4 = v * 4.0f;                      /* exact */
    int quad = (int)q4;                       /* 0..3 */
    float fr = q4 - (float)quad;              /* exact, [0, 1) */
    float phi = fr * 0x1.921fb6p+0f;          /* [0, pi/2) */
    float p2 = phi * phi;
    float sp = 0x1.612462p-33f;               /*  1/13! */
    sp = sp * p2 + -0x1.ae6456p-26f;          /* -1/11! */
    sp = sp * p2 + 0x1.71de3ap-19f;           /*  1/9!  */
    sp = sp * p2 + -0x1.a01a02p-13f;          /* -1/7!  */
    sp = sp * p2 + 0x1.111112p-7f;            /*  1/5!  */
    sp = sp * p2 + -0x1.555556p-3f;           /* -1/3!  */
    float sn = phi + (phi * p2) * sp;
    float cp = -0x1.93974ap-37f;              /* -1/14! */
    cp = cp * p2 + 0x1.1eed8ep-29f;           /*  1/12! */
    cp = cp * p2 + -0x1.27e4fcp-22f;          /* -1/10! */
    cp = cp * p2 + 0x1.a01a02p-16f;           /*  1/8!  */
    cp = cp * p2 + -0x1.6c16c2p-10f;          /* -1/6!  */
    cp = cp * p2 + 0x1.555556p-5f;            /*  1/4!  */
    cp = cp * p2 + -0.5f;                     /* -1/2!  */
    float cs = 1.0f + p2 * cp;
    float c, s;
    switch (quad) {
    case 0:  c = cs;  s = sn;  break;
    case 1:  c = -sn; s = cs;  break;
    case 2:  c = -cs; s = -sn; break;
    default: c = sn;  s = -cs; break;
    }
    *c_out = c; *s_out = s;
}

/* two normals from two raw 32-bit draws */
void wl_box_muller(uint32_t a, uint32_t b, float* z0, float* z1)
{
    float u1 = wl_uniform(a), u2 = wl_uniform(b);
    float r = __builtin_sqrtf(-2.0f * wl_log(u1));
    float c, s;
    wl_sincos2pi(u2, &c, &s);
    *z0 = r * c;
    *z1 = r * s;
}

void wl_normal4(uint64_t seed, uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3, float z[4])
{
    uint32_t ctr[4] = {c0, c1, c2, c3};
    uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    uint32_t r[4];
    wl_philox4x32_10(ctr, key, r);
    wl_box_muller(r[0], r[1], &z[0], &z[1]);
    wl_box_muller(r[2], r[3], &z[2], &z[3]);
}

float wl_student_t3(uint64_t seed, int64_t i, uint32_t t, uint32_t w)
{
    float z[4];
    wl_normal4(seed, (uint32_t)i, (uint32_t)((uint64_t)i >> 32), t, 0x80000000u | w, z);
    float den = (z[1] * z[1] + z[2] * z[2]) + z[3] * z[3];
    den = den / 3.0f;
    return z[0] / __builtin_sqrtf(den);
}

uint16_t wl_bf16_rne(float f)
{
    uint32_t b = u32_from_f32(f);
    uint32_t bias = 0x7FFFu + ((b >> 16) & 1u);
    return (uint16_t)((b + bias) >> 16);
}

/* ---- streams ------------------------------------------------------------ */

/* The four normals of one Philox call of a normal stream, kept while a loop
 * walks the four elements that share the call (q = i / 4).  Only a cache:
 * every value is the one a fresh call would give. */
typedef struct {
    uint64_t q;
    int valid;
    float z[4];
} normal_cache;

/* One gradient value for element i of worker w at step t.  `layer` is the
 * tensor holding i; std/heavy describe it. */
static float grad_value(uint64_t seed, int64_t i, uint32_t t, uint32_t w,
                        float std, int heavy, float heavy_scale, normal_cache* nc)
{
    if (heavy)
        return heavy_scale * wl_student_t3(seed, i, t, w);
    uint64_t q = (uint64_t)i >> 2;
    if (!nc->valid || nc->q != q) {
        wl_normal4(seed, (uint32_t)q, (uint32_t)(q >> 32), t, w, nc->z);
        nc->q = q;
        nc->valid = 1;
    }
    return std * nc->z[i & 3];
}

/* Gradients of worker w at step t for elements [0, N), written to out[0..N).
 * Layer l covers [off[l], off[l] + numel[l]). */
void wl_gen_grads_f32(uint64_t seed, int64_t t, int32_t w, int64_t N, int32_t L,
                      const int64_t* off, const int64_t* numel,
                      const float* std, const uint8_t* heavy, float heavy_scale,
                      float* out)
{
    for (int32_t l = 0; l < L; ++l) {
        int64_t lo = off[l], hi = off[l] + numel[l];
        if (hi > N) hi = N;
        int hv = heavy ? heavy[l] != 0 : 0;
        normal_cache nc = {0, 0, {0.0f, 0.0f, 0.0f, 0.0f}};
        for (int64_t i = lo; i < hi; ++i)
            out[i] = grad_value(seed, i, (uint32_t)t, (uint32_t)w, std[l], hv, heavy_scale, &nc);
    }
}

void wl_gen_grads_bf16(uint64_t seed, int64_t t, int32_t w, int64_t N, int32_t L,
                       const int64_t* off, const int64_t* numel,
                       const float* std, const uint8_t* heavy, float heavy_scale,
                       uint16_t* out)
{
    for (int32_t l = 0; l < L; ++l) {
        int64_t lo = off[l], hi = off[l] + numel[l];
        if (hi > N) hi = N;
        int hv = heavy ? heavy[l] != 0 : 0;
        normal_cache nc = {0, 0, {0.0f, 0.0f, 0.0f, 0.0f}};
        for (int64_t i = lo; i < hi; ++i)
            out[i] = wl_bf16_rne(grad_value(seed, i, (uint32_t)t, (uint32_t)w, std[l], hv, heavy_scale,
                                            &nc));
    }
}

/* Initial parameters: std * Z, stream 0x7FFFFFFF, t = 0, elements [lo, hi). */
void wl_gen_params(uint64_t seed, int64_t lo, int64_t hi, float std, float* out)
{
    uint64_t qz = 0;
    int have = 0;
    float z[4];
    for (int64_t i = lo; i < hi; ++i) {
        uint64_t q = (uint64_t)i >> 2;
        if (!have || q != qz) {
            wl_normal4(seed, (uint32_t)q, (uint32_t)(q >> 32), 0u, 0x7FFFFFFFu, z);
            qz = q;
            have = 1;
        }
        out[i - lo] = std * z[i & 3];
    }
}

/* Gradients of worker w at step t for the flat index range [lo, hi) only,
 * written to out[0 .. hi-lo).  Same values as wl_gen_grads_f32. */
void wl_gen_grads_range_f32(uint64_t seed, int64_t t, int32_t w, int64_t lo, int64_t hi,
                            int32_t L, const int64_t* off, const int64_t* numel,
                            const float* std, const uint8_t* heavy, float heavy_scale,
                            float* out)
{
    int32_t l = 0;
    normal_cache nc = {0, 0, {0.0f, 0.0f, 0.0f, 0.0f}};
    for (int64_t i = lo; i < hi; ++i) {
        while (l < L - 1 && i >= off[l] + numel[l]) ++l;
        int hv = heavy ? heavy[l] != 0 : 0;
        out[i - lo] = grad_value(seed, i, (uint32_t)t, (uint32_t)w, std[l], hv, heavy_scale, &nc);
    }
}
