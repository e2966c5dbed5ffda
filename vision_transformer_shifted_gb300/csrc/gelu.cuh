// The exact GELU of the Swin block's MLP, for the GEMM epilogues and the fused
// MLP kernel.
#pragma once

namespace swin {

// GELU(x) = x Phi(x) = x (1 + erf(x / sqrt 2)) / 2 with erf(u) from an odd
// polynomial u P(u^2) fitted for this library: a weighted least-squares fit
// of erf(u)/u in the Chebyshev basis over u^2 in [0, 3.7^2] (degree 12, weight
// u, float64), rewritten as a power series in s = 2 u^2 / 3.7^2 - 1 and
// evaluated by Horner in fp32; erf = sign(u) beyond |u| = 3.7 (1 - erf(3.7) =
// 1.7e-7).  Measured against float64 erf on 800,001 points in [-8, 8]: erf
// error <= 9.9e-7, GELU error <= 2.8e-6 -- far below the bf16 rounding of the
// result -- in 13 FMAs and no special-function unit instruction.
__device__ __forceinline__ float gelu_poly(float x)
{
    const float u = x * 0.70710678118654752f, t = u * u;
    const float s = fmaf(t, 0.14609204f, -1.0f);
    float p = 3.387000179e-03f;
    p = fmaf(p, s, -8.247348480e-03f);
    p = fmaf(p, s, 6.714036223e-03f);
    p = fmaf(p, s, -8.770867251e-03f);
    p = fmaf(p, s, 2.361703850e-02f);
    p = fmaf(p, s, -3.920292482e-02f);
    p = fmaf(p, s, 5.219075084e-02f);
    p = fmaf(p, s, -6.962815672e-02f);
    p = fmaf(p, s, 9.047554433e-02f);
    p = fmaf(p, s, -1.127380058e-01f);
    p = fmaf(p, s, 1.408007443e-01f);
    p = fmaf(p, s, -1.904647499e-01f);
    p = fmaf(p, s, 3.821373880e-01f);
    const float e = t < 13.69f ? u * p : copysignf(1.0f, u);
    return 0.5f * x * (1.0f + e);
}

// The same for two values at once, on two-lane fp32 instructions (fma.rn.f32x2
// and friends): the same polynomial, the same operations per value.
__device__ __forceinline__ void gelu_poly2(float &x0, float &x1)
{
    float u0 = x0, u1 = x1;
    asm("{\n\t.reg .b64 u, c;\n\tmov.b64 u, {%0, %1};\n\tmov.b64 c, {%2, %2};\n\t"
        "mul.rn.f32x2 u, u, c;\n\tmov.b64 {%0, %1}, u;\n\t}"
        : "+f"(u0), "+f"(u1)
        : "f"(0.70710678118654752f));
    float t0 = u0, t1 = u1;
    asm("{\n\t.reg .b64 t;\n\tmov.b64 t, {%0, %1};\n\tmul.rn.f32x2 t, t, t;\n\tmov.b64 {%0, %1}, t;\n\t}"
        : "+f"(t0), "+f"(t1));
    float s0 = t0, s1 = t1;
    asm("{\n\t.reg .b64 s, a, b;\n\tmov.b64 s, {%0, %1};\n\tmov.b64 a, {%2, %2};\n\tmov.b64 b, {%3, %3};\n\t"
        "fma.rn.f32x2 s, s, a, b;\n\tmov.b64 {%0, %1}, s;\n\t}"
        : "+f"(s0), "+f"(s1)
        : "f"(0.14609204f), "f"(-1.0f));
    static constexpr float k[13] = {3.387000179e-03f, -8.247348480e-03f, 6.714036223e-03f, -8.770867251e-03f,
                                    2.361703850e-02f, -3.920292482e-02f, 5.219075084e-02f, -6.962815672e-02f,
                                    9.047554433e-02f, -1.127380058e-01f, 1.408007443e-01f, -1.904647499e-01f,
                                    3.821373880e-01f};
    float p0 = k[0], p1 = k[0];
#pragma unroll
    for (int i = 1; i < 13; ++i)
        asm("{\n\t.reg .b64 p, s, c;\n\tmov.b64 p, {%0, %1};\n\tmov.b64 s, {%2, %3};\n\tmov.b64 c, {%4, %4};\n\t"
            "fma.rn.f32x2 p, p, s, c;\n\tmov.b64 {%0, %1}, p;\n\t}"
            : "+f"(p0), "+f"(p1)
            : "f"(s0), "f"(s1), "f"(k[i]));
    const float e0 = t0 < 13.69f ? u0 * p0 : copysignf(1.0f, u0);
    const float e1 = t1 < 13.69f ? u1 * p1 : copysignf(1.0f, u1);
    x0 = 0.5f * x0 * (1.0f + e0);
    x1 = 0.5f * x1 * (1.0f + e1);
}

} // namespace swin
