// The fused optimizer step of the MXFP8 variant.
//
// "面向 Blockwise FP8 量化的 ZeRO 优化器设计" §Blockwise 量化: MXFP8 is the
// Blackwell format that gives every memory-contiguous block its own E8M0
// scale (OCP Microscaling specification v1.0); §Blockwise 量化给 ZeRO-1 带来的
// 挑战: such blocks survive a flat ZeRO split, so no fold is needed.  The
// shard is a flat run of the params' row-major elements; a group of 32
// consecutive values shares the scale X = 2^(floor(log2 amax) - 8), clamped to
// 2^-127 .. 2^127 (X = 1 when amax = 0), stored as the E8M0 code
// log2(X) + 127, and each value becomes E4M3(p / X), rounded to nearest even
// and saturated at 448.  The update is update.cuh's, bit for bit the
// block-wise one.  There is no table and no CTA barrier: a group is 8
// consecutive lanes (one float4 each), its amax three shuffles.
//
// Work split: a warp tile is 128 consecutive chunks (2 KB of each FP32
// array); each CTA takes its own run of 32 consecutive tiles, its 8 warps on
// consecutive tiles (4 each), 2 CTAs resident per SM.  Runs of 16 to 64
// tiles were within about 1% of each other on buffers of 88 M to 1.41 G
// elements; 8 (one tile per warp) lost 8-15% and 512 up to 30%.  A persistent
// grid-stride loop (8 CTAs per SM over the whole buffer) ran the MoE buffer
// in 6.08-6.11 ms on some GB300s and 6.45 ms on others; this split ran it in
// 5.90 ms on one of the latter.
//
// fp8z1_mx_step_select runs the same body with a second scalar set picked by
// a device flag, in its own kernel with its own argument struct (the plain
// kernel's parameters stay what it reads).
#include "update.cuh"

namespace {

using namespace fp8z1;

constexpr int kMxThreads = 256;
struct MxArgs {
    const float4* grad;
    float4* master;
    float4* mom1;
    float4* mom2;
    uint32_t* codes;
    uint8_t* scales;   // one E8M0 code per group
    const double* sumsq;
    const int32_t* found_inf;
    int64_t n_chunks;  // float4 chunks: 8 per group
    StepScalars c;
};

// The select kernel's arguments: the plain step's, the second scalar set and
// the flag that picks it (kept apart from MxArgs, whose layout the plain
// kernel's code generation is tuned on).
struct MxSelArgs {
    MxArgs a;
    const int32_t* select;  // a.c when *select == 0, else c2
    StepScalars c2;
};

// A warp tile is kMxUnroll x 32 consecutive chunks (for each u, the 32 lanes
// hold 4 whole groups); the warp issues every load of a tile before any
// update: with 2 CTAs resident per SM (16 warps) about 128 KB of loads in
// flight per SM.
constexpr int kMxUnroll = 4;
constexpr int kMxTile = 32 * kMxUnroll;  // chunks
constexpr int64_t kMxTilesPerCta = 32;

// The update and quantise of this CTA's run of tiles, with the scalars c.
__device__ __forceinline__ void mx_body(const MxArgs& a, const StepScalars& c, float gs)
{
    const int lane = threadIdx.x & 31;
    const int64_t ntiles = (a.n_chunks + kMxTile - 1) / kMxTile;
    const int64_t t0 = (int64_t)blockIdx.x * ntiles / gridDim.x;
    const int64_t t1 = (int64_t)(blockIdx.x + 1) * ntiles / gridDim.x;
    // the trip count is uniform across a warp, so the group shuffles always see
    // all 32 lanes; a group's 8 lanes are in or out of range together (tiles
    // start at multiples of 8 chunks, and so does the end of the last group)
    for (int64_t t = t0 + (threadIdx.x >> 5); t < t1; t += kMxThreads / 32) {
        const int64_t wbase = t * kMxTile;
        float4 g4[kMxUnroll], p4[kMxUnroll], m4[kMxUnroll], v4[kMxUnroll];
#pragma unroll
        for (int u = 0; u < kMxUnroll; ++u) {
            const int64_t i = wbase + u * 32 + lane;
            if (i < a.n_chunks) {
                g4[u] = __ldcs(a.grad + i);
                p4[u] = a.master[i];
                m4[u] = a.mom1[i];
                v4[u] = a.mom2[i];
            } else {
                g4[u] = p4[u] = m4[u] = v4[u] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
#pragma unroll
        for (int u = 0; u < kMxUnroll; ++u) {
            const int64_t i = wbase + u * 32 + lane;
            const bool valid = i < a.n_chunks;
            if (valid) {
                adamw(gs, c, g4[u].x, p4[u].x, m4[u].x, v4[u].x);
                adamw(gs, c, g4[u].y, p4[u].y, m4[u].y, v4[u].y);
                adamw(gs, c, g4[u].z, p4[u].z, m4[u].z, v4[u].z);
                adamw(gs, c, g4[u].w, p4[u].w, m4[u].w, v4[u].w);
                __stcs(a.mom1 + i, m4[u]);
                __stcs(a.mom2 + i, v4[u]);
                __stcs(a.master + i, p4[u]);
            }
            const float4 p = p4[u];
            float amax = fmaxf(fmaxf(fabsf(p.x), fabsf(p.y)), fmaxf(fabsf(p.z), fabsf(p.w)));
            amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
            amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
            amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 4));
            // floor(log2 amax) - 8 from the exponent field (a subnormal amax has
            // field 0 and clamps to -127); 2^-s is then a normal float
            int sexp = 0;
            if (amax != 0.0f) {
                sexp = (int)((__float_as_uint(amax) >> 23) & 0xffu) - 127 - 8;
                sexp = sexp < -127 ? -127 : (sexp > 127 ? 127 : sexp);
            }
            const float inv = __uint_as_float((uint32_t)(127 - sexp) << 23);
            const uint32_t lo = e4m3x2(__fmul_rn(p.x, inv), __fmul_rn(p.y, inv));
            const uint32_t hi = e4m3x2(__fmul_rn(p.z, inv), __fmul_rn(p.w, inv));
            if (valid) __stcs(a.codes + i, lo | (hi << 16));
            // the warp's four group scales as one streaming 4-byte store when
            // aligned and all real (four byte stores of the default policy left
            // the scales' lines in L2 and cost the step 1%)
            const uint32_t e8 = (uint32_t)(sexp + 127);
            const uint32_t b1 = __shfl_sync(0xffffffffu, e8, 8), b2 = __shfl_sync(0xffffffffu, e8, 16),
                           b3 = __shfl_sync(0xffffffffu, e8, 24);
            const bool all4 = __shfl_sync(0xffffffffu, valid ? 1 : 0, 24) != 0;
            uint8_t* sdst = a.scales + (i >> 3);
            if (all4 && (reinterpret_cast<uintptr_t>(a.scales + ((wbase + u * 32) >> 3)) & 3) == 0) {
                if (lane == 0) __stcs(reinterpret_cast<unsigned int*>(sdst), e8 | (b1 << 8) | (b2 << 16) | (b3 << 24));
            } else if (valid && (lane & 7) == 0) {
                *sdst = (uint8_t)e8;
            }
        }
    }
}

// Scalars by value (the plain step).
__global__ void __launch_bounds__(kMxThreads, 2) mx_step_kernel(const MxArgs a)
{
    if (*a.found_inf != 0) return;  // skipped step: write nothing
    __shared__ float s_gscale;
    if (threadIdx.x == 0) s_gscale = grad_factor(*a.sumsq, a.c);
    __syncthreads();
    mx_body(a, a.c, s_gscale);
}

// Two scalar sets by value, picked by *select behind one uniform branch.
__global__ void __launch_bounds__(kMxThreads, 2) mx_step_kernel_select(const MxSelArgs sa)
{
    if (*sa.a.found_inf != 0) return;  // skipped step: write nothing
    __shared__ float s_gscale;
    __shared__ int s_alt;
    if (threadIdx.x == 0) {
        const bool alt = *sa.select != 0;
        s_alt = alt;
        s_gscale = grad_factor(*sa.a.sumsq, alt ? sa.c2 : sa.a.c);
    }
    __syncthreads();
    if (s_alt)
        mx_body(sa.a, sa.c2, s_gscale);
    else
        mx_body(sa.a, sa.a.c, s_gscale);
}

int mx_step_impl(const fp8z1_mx_layout* L, const fp8z1_adamw_hp* hp, const fp8z1_adamw_hp* hp_if_set,
                 const int32_t* d_select, const float* grad_shard, float* master_shard, float* m_shard,
                 float* v_shard, uint8_t* fp8_shard, uint8_t* scale_shard, int64_t g0, int64_t g1,
                 const double* d_sumsq, const int32_t* d_found_inf, void* stream)
{
    if (!L || !hp || !grad_shard || !master_shard || !m_shard || !v_shard || !fp8_shard || !scale_shard ||
        !d_sumsq || !d_found_inf || !in_domain(hp) || (hp_if_set && !in_domain(hp_if_set)))
        return FP8Z1_EINVAL;
    if ((hp_if_set == nullptr) != (d_select == nullptr)) return FP8Z1_EINVAL;
    if (g0 < 0 || g1 < g0 || g1 > L->n_groups) return FP8Z1_EINVAL;
    if (!L->on_device) return FP8Z1_ENODEV;
    if (!fp8z1::aligned(grad_shard, 16) || !fp8z1::aligned(master_shard, 16) || !fp8z1::aligned(m_shard, 16) ||
        !fp8z1::aligned(v_shard, 16) || !fp8z1::aligned(fp8_shard, 16) || !fp8z1::aligned(d_sumsq, 8) ||
        !fp8z1::aligned(d_found_inf, 4) || (d_select && !fp8z1::aligned(d_select, 4)))
        return FP8Z1_EALIGN;
    const int64_t chunks = (g1 - g0) * (FP8Z1_MX_GROUP / 4);
    if (chunks == 0) return FP8Z1_OK;
    MxArgs a = {};
    a.grad = reinterpret_cast<const float4*>(grad_shard);
    a.master = reinterpret_cast<float4*>(master_shard);
    a.mom1 = reinterpret_cast<float4*>(m_shard);
    a.mom2 = reinterpret_cast<float4*>(v_shard);
    a.codes = reinterpret_cast<uint32_t*>(fp8_shard);
    a.scales = scale_shard;
    a.sumsq = d_sumsq;
    a.found_inf = d_found_inf;
    a.n_chunks = chunks;
    a.c = scalars(hp);
    // runs of 32 tiles; a buffer too small to give every SM two such CTAs gets
    // runs of one tile per warp (or fewer CTAs) instead
    const int64_t ntiles = (chunks + kMxTile - 1) / kMxTile;
    int64_t grid = (ntiles + kMxTilesPerCta - 1) / kMxTilesPerCta;
    if (grid < 2 * (int64_t)L->sm_count) {
        const int64_t per_warp = (ntiles + kMxThreads / 32 - 1) / (kMxThreads / 32);
        grid = per_warp < 2 * (int64_t)L->sm_count ? per_warp : 2 * (int64_t)L->sm_count;
    }
    fp8z1::count_launch();
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (d_select) {
        MxSelArgs sa = {};
        sa.a = a;
        sa.select = d_select;
        sa.c2 = scalars(hp_if_set);
        mx_step_kernel_select<<<(unsigned)grid, kMxThreads, 0, s>>>(sa);
    } else {
        mx_step_kernel<<<(unsigned)grid, kMxThreads, 0, s>>>(a);
    }
    return fp8z1::launch_status();
}

}  // namespace

extern "C" int fp8z1_mx_step_select(const fp8z1_mx_layout* L, const fp8z1_adamw_hp* hp_if_clear,
                                    const fp8z1_adamw_hp* hp_if_set, const int32_t* d_select,
                                    const float* grad_shard, float* master_shard, float* m_shard, float* v_shard,
                                    uint8_t* fp8_shard, uint8_t* scale_shard, int64_t g0, int64_t g1,
                                    const double* d_sumsq, const int32_t* d_found_inf, void* stream)
{
    fp8z1::NvtxRange nvtx_range("fp8z1_mx_step_select");
    if (!hp_if_set || !d_select) return FP8Z1_EINVAL;
    return mx_step_impl(L, hp_if_clear, hp_if_set, d_select, grad_shard, master_shard, m_shard, v_shard, fp8_shard,
                        scale_shard, g0, g1, d_sumsq, d_found_inf, stream);
}

extern "C" int fp8z1_mx_step(const fp8z1_mx_layout* L, const fp8z1_adamw_hp* hp, const float* grad_shard,
                             float* master_shard, float* m_shard, float* v_shard, uint8_t* fp8_shard,
                             uint8_t* scale_shard, int64_t g0, int64_t g1, const double* d_sumsq,
                             const int32_t* d_found_inf, void* stream)
{
    fp8z1::NvtxRange nvtx_range("fp8z1_mx_step");
    return mx_step_impl(L, hp, nullptr, nullptr, grad_shard, master_shard, m_shard, v_shard, fp8_shard, scale_shard,
                        g0, g1, d_sumsq, d_found_inf, stream);
}
