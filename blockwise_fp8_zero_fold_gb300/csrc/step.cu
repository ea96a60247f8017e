// The fused optimizer step over a block range of the shard: unscale + clip +
// AdamW on the FP32 master/m/v, then the block's scale and E4M3 codes, in one
// HBM pass.
//
// "面向 Blockwise FP8 量化的 ZeRO 优化器设计" §总结: the optimizer update is
// elementwise on the rank's slice, and each rank then quantises new FP8 params
// and their scales from its FP32 master; §Blockwise 量化: one scale per
// 128x128 block.  "DeepSpeed ZeRO 优化" §三: unscale and clip, then the
// update, then the low-precision copy; §七: clip_coef = max_norm /
// (||g_s|| / S + 1e-6), applied when < 1; §六: a found inf skips the step.
//
// One CTA of 512 threads per block of 16384 elements; thread t owns the
// float4 chunks t, t+512, ..., t+3584 of the block.  It streams grad / master
// / m / v in, updates them, writes master / m / v back at once and keeps its
// 32 new master values in registers while the CTA reduces the block amax
// (warp shuffles, then 16 partials in shared memory).  The codes are then
// produced from the registers: no second pass over HBM.
//
// FP32 operation order per element (no contraction beyond the explicit fmas;
// division and square root correctly rounded):
//   g   = g_s * gscale,  gscale = (clip_coef < 1 ? (float)clip_coef : 1) / S
//   m   = fma(beta1, m, (1-beta1) * g)
//   v   = fma(beta2, v, ((1-beta2) * g) * g)
//   den = fma(sqrt(v), 1/sqrt(1-beta2^t), eps)
//   p   = fma(-lr/(1-beta1^t), m / den, p * (1 - lr*wd))
// scale = amax/448 (1 when amax == 0); code = cvt.rn.satfinite.e4m3(p / scale).
#include <math.h>

#include "internal.h"

namespace {

constexpr int kThreads = 512;
constexpr int kVec = FP8Z1_BLOCK_ELEMS / 4 / kThreads;  // 8 float4 per thread
constexpr int kWarps = kThreads / 32;

struct StepScalars {
    float beta1, beta2, omb1, omb2, eps, step_size, inv_sqrt_bc2, decay, max_norm, loss_scale;
};

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

__device__ __forceinline__ float warp_max(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

__global__ void __launch_bounds__(kThreads, 2) step_kernel(const float4* __restrict__ grad,
                                                           float4* __restrict__ master,
                                                           float4* __restrict__ mom1,
                                                           float4* __restrict__ mom2,
                                                           uint32_t* __restrict__ codes,
                                                           float* __restrict__ scales,
                                                           const double* __restrict__ d_sumsq,
                                                           const int32_t* __restrict__ d_found_inf,
                                                           StepScalars c)
{
    if (*d_found_inf != 0) return;  // skipped step: write nothing
    __shared__ float s_gscale;
    __shared__ float s_amax[kWarps];
    const int tid = threadIdx.x;
    if (tid == 0) {
        const double global = sqrt(*d_sumsq) / (double)c.loss_scale;
        const double coef = (double)c.max_norm / (global + 1e-6);
        const float clip = coef < 1.0 ? (float)coef : 1.0f;
        s_gscale = __fdiv_rn(clip, c.loss_scale);
    }
    __syncthreads();
    const float gs = s_gscale;

    const int64_t base = (int64_t)blockIdx.x * (FP8Z1_BLOCK_ELEMS / 4) + tid;
    float pn[4 * kVec];
    float amax = 0.0f;
#pragma unroll
    for (int j = 0; j < kVec; ++j) {
        const int64_t i = base + j * kThreads;
        const float4 g4 = __ldcs(grad + i);
        float4 p4 = master[i];
        float4 m4 = mom1[i];
        float4 v4 = mom2[i];
        adamw(gs, c, g4.x, p4.x, m4.x, v4.x);
        adamw(gs, c, g4.y, p4.y, m4.y, v4.y);
        adamw(gs, c, g4.z, p4.z, m4.z, v4.z);
        adamw(gs, c, g4.w, p4.w, m4.w, v4.w);
        __stcs(mom1 + i, m4);
        __stcs(mom2 + i, v4);
        __stcs(master + i, p4);
        pn[4 * j + 0] = p4.x;
        pn[4 * j + 1] = p4.y;
        pn[4 * j + 2] = p4.z;
        pn[4 * j + 3] = p4.w;
        amax = fmaxf(amax, fmaxf(fmaxf(fabsf(p4.x), fabsf(p4.y)), fmaxf(fabsf(p4.z), fabsf(p4.w))));
    }

    amax = warp_max(amax);
    if ((tid & 31) == 0) s_amax[tid >> 5] = amax;
    __syncthreads();
    float bmax = s_amax[0];
#pragma unroll
    for (int w = 1; w < kWarps; ++w) bmax = fmaxf(bmax, s_amax[w]);
    const float scale = bmax == 0.0f ? 1.0f : __fdiv_rn(bmax, 448.0f);
    if (tid == 0) scales[blockIdx.x] = scale;

#pragma unroll
    for (int j = 0; j < kVec; ++j) {
        const uint32_t lo = e4m3x2(__fdiv_rn(pn[4 * j + 0], scale), __fdiv_rn(pn[4 * j + 1], scale));
        const uint32_t hi = e4m3x2(__fdiv_rn(pn[4 * j + 2], scale), __fdiv_rn(pn[4 * j + 3], scale));
        __stcs(codes + base + j * kThreads, lo | (hi << 16));
    }
}

bool in_domain(const fp8z1_adamw_hp* hp)
{
    return hp->step >= 1 && hp->lr >= 0.0f && hp->beta1 >= 0.0f && hp->beta1 < 1.0f &&
           hp->beta2 >= 0.0f && hp->beta2 < 1.0f && hp->eps > 0.0f && hp->weight_decay >= 0.0f &&
           hp->max_norm > 0.0f && hp->loss_scale > 0.0f && isfinite(hp->loss_scale) &&
           isfinite(hp->lr) && isfinite(hp->eps) && isfinite(hp->weight_decay);
}

}  // namespace

extern "C" int fp8z1_step(const fp8z1_layout* L, const fp8z1_adamw_hp* hp, const float* grad_shard,
                          float* master_shard, float* m_shard, float* v_shard, uint8_t* fp8_shard,
                          float* scale_shard, int64_t b0, int64_t b1, const double* d_sumsq,
                          const int32_t* d_found_inf, void* stream)
{
    if (!hp || !grad_shard || !master_shard || !m_shard || !v_shard || !fp8_shard || !scale_shard ||
        !d_sumsq || !d_found_inf || !in_domain(hp))
        return FP8Z1_EINVAL;
    const int st = fp8z1::check_range(L, b0, b1);
    if (st != FP8Z1_OK) return st;
    if (b1 - b0 > 0x7fffffffLL) return FP8Z1_EINVAL;
    if (!fp8z1::aligned(grad_shard, 16) || !fp8z1::aligned(master_shard, 16) ||
        !fp8z1::aligned(m_shard, 16) || !fp8z1::aligned(v_shard, 16) || !fp8z1::aligned(fp8_shard, 16) ||
        !fp8z1::aligned(scale_shard, 4) || !fp8z1::aligned(d_sumsq, 8) || !fp8z1::aligned(d_found_inf, 4))
        return FP8Z1_EALIGN;
    if (b0 == b1) return FP8Z1_OK;

    // per-step scalars, in double on the host, rounded once to FP32
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

    step_kernel<<<(unsigned)(b1 - b0), kThreads, 0, static_cast<cudaStream_t>(stream)>>>(
        reinterpret_cast<const float4*>(grad_shard), reinterpret_cast<float4*>(master_shard),
        reinterpret_cast<float4*>(m_shard), reinterpret_cast<float4*>(v_shard),
        reinterpret_cast<uint32_t*>(fp8_shard), scale_shard, d_sumsq, d_found_inf, c);
    return fp8z1::launch_status();
}
