// Packed binary32 pairs (Blackwell add / sub / mul .rn.f32x2): one
// instruction performs the same operation on two independent binary32
// values, each lane an IEEE operation rounded to nearest even with subnormals
// kept -- the same bits as the scalar __fadd_rn / __fsub_rn / __fmul_rn.  The
// kernels use them where two independent operations of the arithmetic stand
// side by side, which halves their issue slots without changing a result.
//
// One rule keeps every operation separately rounded: the code generator may
// fuse a packed multiply with a packed add or subtract that consumes its
// result into one fused multiply-add (measured on sm_103a, also with fmad
// contraction switched off), but it never fuses explicitly rounded scalar
// operations.  So a packed product is only ever consumed by scalar adds (or
// by multiplies, conversions, stores), and a packed add or subtract only
// takes scalar products, sums, loads or selects.  The bit-exact parity tests
// would catch a sequence that breaks it.
#pragma once
#include <cuda_runtime.h>

namespace lamb1b {

__device__ __forceinline__ float2 fadd2(float2 a, float2 b)
{
    float2 r;
    asm("{\n\t.reg .b64 pa, pb, pr;\n\t"
        "mov.b64 pa, {%2, %3};\n\tmov.b64 pb, {%4, %5};\n\t"
        "add.rn.f32x2 pr, pa, pb;\n\t"
        "mov.b64 {%0, %1}, pr;\n\t}"
        : "=f"(r.x), "=f"(r.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return r;
}

__device__ __forceinline__ float2 fsub2(float2 a, float2 b)
{
    float2 r;
    asm("{\n\t.reg .b64 pa, pb, pr;\n\t"
        "mov.b64 pa, {%2, %3};\n\tmov.b64 pb, {%4, %5};\n\t"
        "sub.rn.f32x2 pr, pa, pb;\n\t"
        "mov.b64 {%0, %1}, pr;\n\t}"
        : "=f"(r.x), "=f"(r.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return r;
}

__device__ __forceinline__ float2 fmul2(float2 a, float2 b)
{
    float2 r;
    asm("{\n\t.reg .b64 pa, pb, pr;\n\t"
        "mov.b64 pa, {%2, %3};\n\tmov.b64 pb, {%4, %5};\n\t"
        "mul.rn.f32x2 pr, pa, pb;\n\t"
        "mov.b64 {%0, %1}, pr;\n\t}"
        : "=f"(r.x), "=f"(r.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return r;
}

__device__ __forceinline__ float2 splat2(float v) { return make_float2(v, v); }

// r[c] = a[c] op b[c] for four consecutive values, as two packed pairs
__device__ __forceinline__ void add4(float (&r)[4], const float (&a)[4], const float (&b)[4])
{
    const float2 lo = fadd2(make_float2(a[0], a[1]), make_float2(b[0], b[1]));
    const float2 hi = fadd2(make_float2(a[2], a[3]), make_float2(b[2], b[3]));
    r[0] = lo.x; r[1] = lo.y; r[2] = hi.x; r[3] = hi.y;
}

__device__ __forceinline__ void sub4(float (&r)[4], const float (&a)[4], const float (&b)[4])
{
    const float2 lo = fsub2(make_float2(a[0], a[1]), make_float2(b[0], b[1]));
    const float2 hi = fsub2(make_float2(a[2], a[3]), make_float2(b[2], b[3]));
    r[0] = lo.x; r[1] = lo.y; r[2] = hi.x; r[3] = hi.y;
}

__device__ __forceinline__ void mul4(float (&r)[4], const float (&a)[4], const float (&b)[4])
{
    const float2 lo = fmul2(make_float2(a[0], a[1]), make_float2(b[0], b[1]));
    const float2 hi = fmul2(make_float2(a[2], a[3]), make_float2(b[2], b[3]));
    r[0] = lo.x; r[1] = lo.y; r[2] = hi.x; r[3] = hi.y;
}

// r[c] = a[c] + b[c] for a pair (scalar adds, so a packed product may feed them)
__device__ __forceinline__ float2 fadd_lanes(float2 a, float2 b)
{
    return make_float2(__fadd_rn(a.x, b.x), __fadd_rn(a.y, b.y));
}

// r[c] = s * a[c]
__device__ __forceinline__ void mul4s(float (&r)[4], float s, const float (&a)[4])
{
    const float2 lo = fmul2(splat2(s), make_float2(a[0], a[1]));
    const float2 hi = fmul2(splat2(s), make_float2(a[2], a[3]));
    r[0] = lo.x; r[1] = lo.y; r[2] = hi.x; r[3] = hi.y;
}

// r[c] = a[c] + s
__device__ __forceinline__ void add4s(float (&r)[4], const float (&a)[4], float s)
{
    const float2 lo = fadd2(make_float2(a[0], a[1]), splat2(s));
    const float2 hi = fadd2(make_float2(a[2], a[3]), splat2(s));
    r[0] = lo.x; r[1] = lo.y; r[2] = hi.x; r[3] = hi.y;
}

}  // namespace lamb1b
