/*
 * lamb1b_gen: on-device generation of the seeded synthetic workload (C ABI).
 *
 * Not part of the optimizer: these calls fill device buffers with initial
 * parameters and per-(worker, step, element) gradients so that benchmarks and
 * tests can run at full size without host traffic.  The same definition is
 * used for gradients drawn inside the optimizer kernels (LAMB1B_GRAD_PHILOX).
 *
 * Definition (binary32, one rounding per operation, no fused multiply-add;
 * how the device evaluates it without changing a bit: lamb1b_gen_selfcheck):
 *   key = (seed lo32, seed hi32); Philox4x32-10 (Salmon et al., "Parallel
 *   random numbers: as easy as 1, 2, 3", SC'11).
 *   uniform(u) = (2*(u >> 9) + 1) * 2^-24.
 *   Box-Muller pairs from outputs (0,1) and (2,3) of one Philox call, with ln
 *   evaluated as e*ln2 + 2 atanh-series(s), s = (f-1)/(f+1), f in
 *   [sqrt(1/2), sqrt(2)], and sin/cos of 2*pi*v by quadrant split and Taylor
 *   series to degree 13/14 (constants and evaluation order as in the
 *   workload generator's reference text).
 *   Normal element i: output i%4 of counter (i/4 lo, i/4 hi, t, w).
 *   Student-t(3) element i: counter (i lo, i hi, t, 0x80000000|w), normals
 *   Z0..Z3, Z0 / sqrt(((Z1^2+Z2^2)+Z3^2)/3).
 *   Parameters: counter (i/4 lo, i/4 hi, 0, 0x7FFFFFFF), std * Z.
 *   bf16: round to nearest even of the binary32 bits.
 *
 * Conventions as in lamb1b.h: device pointers, stream as void*, 0 or a
 * negative LAMB1B_ERR_* code, asynchronous.
 */
#ifndef LAMB1B_GEN_H
#define LAMB1B_GEN_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* out_dev[w*ld + i] for w in [0, W), i in [0, N): gradient of worker w at
 * step t.  Tensor l covers [layer_off[l], layer_off[l] + layer_numel[l]);
 * layer_off, layer_numel, layer_std and layer_heavy are HOST arrays of L
 * entries (layer_heavy may be NULL: no Student-t tensors).  bf16 != 0 writes
 * bfloat16 bit patterns (uint16) instead of binary32.  Elements [N, ld) of
 * each row are left untouched.  ld >= N.  One launch per tensor. */
int lamb1b_gen_grads(void* out_dev, int64_t ld, int32_t W, int32_t bf16,
                     uint64_t seed, int64_t t,
                     const int64_t* layer_off, const int64_t* layer_numel, int32_t L,
                     const float* layer_std, const uint8_t* layer_heavy,
                     float heavy_scale, void* stream);

/* out_dev[j] = parameter lo + j for j in [0, hi - lo). */
int lamb1b_gen_params(float* out_dev, int64_t lo, int64_t hi, float std,
                      uint64_t seed, void* stream);

/* Self-check of how the device evaluates the definition above (a testing
 * hook; no counterpart in the paper).  The device transform packs pairs of
 * binary32 operations into one instruction and computes its divisions by
 * (f+1) and by 3 and its square roots with Markstein's method (approximate
 * reciprocal or reciprocal square root, one Newton-Raphson step, a final
 * correction from the exact remainder), which give the IEEE result on the
 * inputs the transform can produce.  This call enumerates those inputs and
 * writes five mismatch counts (0 means exact) to counts_dev (caller-owned
 * device memory, 5 x uint64, 8-byte aligned; zeroed by the call):
 *   [0] all 2^23 log-series quotients (f-1)/(f+1);
 *   [1] x / 3 for every non-negative binary32 x;
 *   [2] sqrt(x) for every binary32 x >= 2^-102 (the transform's square
 *       roots see x >= 1.19e-7 and, in Student-t, x >= 1.6e-20);
 *   [3] the four normals of 2^22 Philox counters against the same draws
 *       written with the IEEE intrinsics one operation at a time;
 *   [4] the Student-t values of 2^22 elements, likewise.
 * Takes a fraction of a second.  Errors: ARG, ALIGN, CUDA. */
int lamb1b_gen_selfcheck(unsigned long long* counts_dev, uint64_t seed, void* stream);

#ifdef __cplusplus
}
#endif
#endif
