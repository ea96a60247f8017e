// The FP32 update and the E4M3 codec shared by the block-wise and the MXFP8
// step kernels: one definition, so both schemes update master / m / v alike,
// bit for bit.
//
// "DeepSpeed ZeRO 优化" §三: unscale and clip, then the update; §七:
// clip_coef = max_norm / (||g_s|| / S + 1e-6), applied when < 1.  The pages
// give no AdamW equations; the reading is decoupled weight decay with bias
// correction.  FP32 operation order per element (no contraction beyond the
// explicit fmas; division and square root correctly rounded):
//   g   = g_s * gscale,  gscale = (clip_coef < 1 ? (float)clip_coef : 1) / S
//   m   = fma(beta1, m, (1-beta1) * g)
//   v   = fma(beta2, v, ((1-beta2) * g) * g)
//   den = fma(sqrt(v), 1/sqrt(1-beta2^t), eps)
//   p   = fma(-lr/(1-beta1^t), m / den, p * (1 - lr*wd))
// with the per-step scalars formed in double on the host and rounded once.
#pragma once

#include <math.h>

#include "internal.h"

namespace fp8z1 {

using StepScalars = fp8z1_step_scalars;

// The unscale and clip folded into one factor, from the global sum of squares
// of the loss-scaled grads (formed in double, as the host would).
__device__ __forceinline__ float grad_factor(double sumsq, const StepScalars& c)
{
    const double global = sqrt(sumsq) / (double)c.loss_scale;
    const double coef = (double)c.max_norm / (global + 1e-6);
    const float clip = coef < 1.0 ? (float)coef : 1.0f;
    return __fdiv_rn(clip, c.loss_scale);
}

__device__ __forceinline__ void adamw(float gs, const StepScalars& c, float g_s, float& p, float& m,
                                      float& v)
{
    const float g = __fmul_rn(g_s, gs);
    m = __fmaf_rn(c.beta1, m, __fmul_rn(c.omb1, g));
    v = __fmaf_rn(c.beta2, v, __fmul_rn(__fmul_rn(c.omb2, g), g));
    const float den = __fmaf_rn(__fsqrt_rn(v), c.inv_sqrt_bc2, c.eps);
    p = __fmaf_rn(-c.step_size, __fdiv_rn(m, den), __fmul_rn(p, c.decay));
}

// two floats -> two E4M3 codes (lo in the low byte), round to nearest even,
// finite overflow saturated to +-448
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi)
{
    unsigned short r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// two E4M3 codes (low byte -> .x) -> their exact values
__device__ __forceinline__ float2 e4m3x2_decode(uint32_t two)
{
    uint32_t h2;
    asm("{ .reg .b16 t; cvt.u16.u32 t, %1; cvt.rn.f16x2.e4m3x2 %0, t; }" : "=r"(h2) : "r"(two));
    float lo, hi;
    asm("{ .reg .b16 a, b; mov.b32 {a, b}, %2; cvt.f32.f16 %0, a; cvt.f32.f16 %1, b; }"
        : "=f"(lo), "=f"(hi) : "r"(h2));
    return make_float2(lo, hi);
}

inline bool in_domain(const fp8z1_adamw_hp* hp)
{
    return hp->step >= 1 && hp->lr >= 0.0f && hp->beta1 >= 0.0f && hp->beta1 < 1.0f &&
           hp->beta2 >= 0.0f && hp->beta2 < 1.0f && hp->eps > 0.0f && hp->weight_decay >= 0.0f &&
           hp->max_norm > 0.0f && hp->loss_scale > 0.0f && isfinite(hp->loss_scale) &&
           isfinite(hp->lr) && isfinite(hp->eps) && isfinite(hp->weight_decay);
}

// per-step scalars, in double on the host, rounded once to FP32
inline StepScalars scalars(const fp8z1_adamw_hp* hp)
{
    const double t = (double)hp->step;
    const double bc1 = 1.0 - pow((double)hp->beta1, t);
    const double bc2 = 1.0 - pow((double)hp->beta2, t);
    StepScalars c;
    c.beta1 = hp->beta1;
    c.beta2 = hp->beta2;
    c.omb1 = (float)(1.0 - (double)hp->beta1);
    c.omb2 = (float)(1.0 - (double)hp->beta2);
    c.eps = hp->eps;
    c.step_size = (float)((double)hp->lr / bc1);
    c.inv_sqrt_bc2 = (float)(1.0 / sqrt(bc2));
    c.decay = (float)(1.0 - (double)hp->lr * (double)hp->weight_decay);
    c.max_norm = hp->max_norm;
    c.loss_scale = hp->loss_scale;
    return c;
}

}  // namespace fp8z1
