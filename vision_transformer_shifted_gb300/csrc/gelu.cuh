// The exact GELU of the Swin block's MLP, for the GEMM epilogues and the fused
// MLP kernel.
#pragma once

#include "ptx.cuh"

namespace swin {

// GELU(x) = x Phi(x) = x (1 + erf(x / sqrt 2)) / 2, erf by the rational-times-
// exponential form of Abramowitz and Stegun, Handbook of Mathematical
// Functions, 7.1.26 (Hastings): for a >= 0, erf(a) = 1 - t (a1 + t (a2 + t (a3
// + t (a4 + t a5)))) exp(-a^2), t = 1 / (1 + p a), |error| <= 1.5e-7; odd in
// the sign.  In fp32 with the hardware reciprocal and exp2, measured against
// float64 erf on 1,800,001 points in [-9, 9]: erf error <= 5.5e-7, GELU error
// <= 4.7e-7 -- far below the bf16 rounding of the result -- in eleven
// multiply-adds and two special-function instructions.
__device__ __forceinline__ float gelu_exact(float x)
{
    const float u = x * 0.70710678118654752f, a = fabsf(u);
    const float t = rcp_approx(fmaf(0.3275911f, a, 1.0f));
    float q = fmaf(1.061405429f, t, -1.453152027f);
    q = fmaf(q, t, 1.421413741f);
    q = fmaf(q, t, -0.284496736f);
    q = fmaf(q, t, 0.254829592f);
    q *= t;
    const float e = ex2_approx(a * (a * -1.4426950408889634f));   // exp(-a^2)
    const float r = copysignf(fmaf(-q, e, 1.0f), u);               // erf(u)
    const float hx = 0.5f * x;
    return fmaf(hx, r, hx);
}

// f32x2 helpers: d = a * b + c, d = a * b (two lanes, one instruction).
__device__ __forceinline__ void g2_fma(float &d0, float &d1, float a0, float a1, float b0, float b1, float c0, float c1)
{
    asm("{\n\t.reg .b64 a, b, c;\n\tmov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\tmov.b64 c, {%6, %7};\n\t"
        "fma.rn.f32x2 a, a, b, c;\n\tmov.b64 {%0, %1}, a;\n\t}"
        : "=f"(d0), "=f"(d1)
        : "f"(a0), "f"(a1), "f"(b0), "f"(b1), "f"(c0), "f"(c1));
}
__device__ __forceinline__ void g2_mul(float &d0, float &d1, float a0, float a1, float b0, float b1)
{
    asm("{\n\t.reg .b64 a, b;\n\tmov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\t"
        "mul.rn.f32x2 a, a, b;\n\tmov.b64 {%0, %1}, a;\n\t}"
        : "=f"(d0), "=f"(d1)
        : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

// gelu_exact of two values with the same operations on two-lane fp32
// instructions (the polynomial's coefficients negated so that 1 - q e is one
// multiply-add).
__device__ __forceinline__ void gelu_exact2(float &x0, float &x1)
{
    float u0, u1, d0, d1;
    g2_mul(u0, u1, x0, x1, 0.70710678118654752f, 0.70710678118654752f);
    const float a0 = fabsf(u0), a1 = fabsf(u1);
    g2_fma(d0, d1, a0, a1, 0.3275911f, 0.3275911f, 1.0f, 1.0f);
    const float t0 = rcp_approx(d0), t1 = rcp_approx(d1);
    float q0, q1;   // -t (a1 + t (a2 + t (a3 + t (a4 + t a5))))
    g2_fma(q0, q1, t0, t1, -1.061405429f, -1.061405429f, 1.453152027f, 1.453152027f);
    g2_fma(q0, q1, q0, q1, t0, t1, -1.421413741f, -1.421413741f);
    g2_fma(q0, q1, q0, q1, t0, t1, 0.284496736f, 0.284496736f);
    g2_fma(q0, q1, q0, q1, t0, t1, -0.254829592f, -0.254829592f);
    g2_mul(q0, q1, q0, q1, t0, t1);
    float z0, z1;
    g2_mul(z0, z1, a0, a1, -1.4426950408889634f, -1.4426950408889634f);
    g2_mul(z0, z1, z0, z1, a0, a1);
    const float e0 = ex2_approx(z0), e1 = ex2_approx(z1);   // exp(-a^2)
    float r0, r1;
    g2_fma(r0, r1, q0, q1, e0, e1, 1.0f, 1.0f);   // erf(|u|)
    r0 = copysignf(r0, u0);
    r1 = copysignf(r1, u1);
    float h0, h1;
    g2_mul(h0, h1, x0, x1, 0.5f, 0.5f);
    g2_fma(x0, x1, h0, h1, r0, r1, h0, h1);
}

} // namespace swin
