// The fused optimizer step over a block range of the shard: unscale + clip +
// AdamW on the FP32 master/m/v, then the block's scale and E4M3 codes, in one
// HBM pass.
//
// "面向 Blockwise FP8 量化的 ZeRO 优化器设计" §总结: the optimizer update is
// elementwise on the rank's slice, and each rank then quantises new FP8 params
// and their scales from its FP32 master; §Blockwise 量化: one scale per
// 128x128 block; §参数布局变换: grads are folded to the optimizer's layout and
// the FP8 params unfolded back.  "DeepSpeed ZeRO 优化" §三: unscale and clip,
// then the update, then the low-precision copy; §七: clip_coef = max_norm /
// (||g_s|| / S + 1e-6), applied when < 1; §六: a found inf skips the step.
//
// One CTA of 512 threads per block of 16384 elements; thread t owns the
// float4 chunks t, t+512, ..., t+3584 of the block (chunk i is row i/32,
// columns 4*(i%32) .. +3 of the 128x128 block, so a warp covers one block row).
// It streams grad / master / m / v in, updates them, writes master / m / v back
// at once and keeps its 32 new master values in registers while the CTA
// reduces the block amax (warp shuffles, then 16 partials in shared memory).
// The codes are then produced from the registers: no second pass over HBM.
//
// Where the grads come from and where the codes go is chosen at compile time:
//   GRAD_ROWS    grads are read from the row-major params through the block
//                lookup table (the fold of the grads, fused), else from the
//                folded grad shard;
//   CODES_ROWS   codes are written into the row-major FP8 params through the
//                lookup table (the unfold of the codes, fused);
//   CODES_FOLDED codes are written to the folded code shard.
//
// The FP32 update is update.cuh's; then scale = amax/448 (1 when amax == 0)
// and code = cvt.rn.satfinite.e4m3(p / scale).
#include <math.h>

#include "update.cuh"

namespace {

using namespace fp8z1;

constexpr int kThreads = 512;
constexpr int kVec = FP8Z1_BLOCK_ELEMS / 4 / kThreads;  // 8 float4 per thread
constexpr int kWarps = kThreads / 32;

struct StepArgs {
    const float4* grad;          // folded grad shard (!GRAD_ROWS)
    float4* master;
    float4* mom1;
    float4* mom2;
    uint32_t* codes;             // folded code shard (CODES_FOLDED)
    float* scales;
    const double* sumsq;
    const int32_t* found_inf;
    const fp8z1_block* lut;      // GRAD_ROWS / CODES_ROWS
    int64_t b0;
    const float* const* grad_params;  // GRAD_ROWS: row-major FP32 grads
    uint8_t* const* code_params;      // CODES_ROWS: row-major FP8 params
    unsigned* status;
    float* block_cos;            // MON: cosine(master, dequantised) per block
    uint32_t* block_underflow;   // MON: non-zero masters whose code is 0, per block
    const StepScalars* dsc;      // DEVSC: the scalars in device memory
    StepScalars c;               // !DEVSC: the scalars by value
};

__device__ __forceinline__ float warp_max(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// the 4 grads of chunk (r, c) of a row-major tile; zeros outside the real extent
__device__ __forceinline__ float4 load_grad_rows(const float* tile, int64_t ld, int r, int c, int rows,
                                                 int cols, bool vec)
{
    float4 g = make_float4(0.f, 0.f, 0.f, 0.f);
    if (r < rows) {
        const float* src = tile + r * ld + c;
        if (vec) {  // ld % 4 == 0: a 4-column group is all real or all padding
            if (c < cols) g = __ldcs(reinterpret_cast<const float4*>(src));
        } else {
            if (c + 0 < cols) g.x = __ldcs(src + 0);
            if (c + 1 < cols) g.y = __ldcs(src + 1);
            if (c + 2 < cols) g.z = __ldcs(src + 2);
            if (c + 3 < cols) g.w = __ldcs(src + 3);
        }
    }
    return g;
}

__device__ __forceinline__ void store_codes_rows(uint8_t* tile, int64_t ld, int r, int c, int rows,
                                                 int cols, bool vec, uint32_t q)
{
    if (r >= rows) return;
    uint8_t* dst = tile + r * ld + c;
    if (vec) {
        if (c < cols) __stcs(reinterpret_cast<unsigned int*>(dst), q);
    } else {
#pragma unroll
        for (int b = 0; b < 4; ++b)
            if (c + b < cols) dst[b] = (uint8_t)(q >> (8 * b));
    }
}

// Quantisation monitors ("FP8训练技术与万亿参数模型优化实践" §1.2: underflow =
// zeros / total, distortion = cosine(original, dequantised)), per block: the
// count of non-zero new masters whose code decodes to 0, and
// sum(p d) / sqrt(sum(p^2) sum(d^2)) with d = decode(code) * scale (1 when both
// are all zero, 0 when only one is).  FP32 sums per thread, double across the
// CTA: a diagnostic, not bit-exact.
__device__ __forceinline__ void monitor_add(float p, float dec, float scale, float& pd, float& pp,
                                            float& dd, uint32_t& under)
{
    const float d = __fmul_rn(dec, scale);
    pd = __fmaf_rn(p, d, pd);
    pp = __fmaf_rn(p, p, pp);
    dd = __fmaf_rn(d, d, dd);
    under += (p != 0.0f && dec == 0.0f) ? 1u : 0u;
}

template <bool GRAD_ROWS, bool CODES_ROWS, bool CODES_FOLDED, bool MON, bool DEVSC>
__global__ void __launch_bounds__(kThreads, 2) step_kernel(const StepArgs a)
{
    if (*a.found_inf != 0) return;  // skipped step: write nothing
    __shared__ float s_gscale;
    __shared__ float s_amax[kWarps];
    __shared__ StepScalars s_c;
    const int tid = threadIdx.x;
    if (tid == 0) {
        if (DEVSC) s_c = *a.dsc;
        s_gscale = grad_factor(*a.sumsq, DEVSC ? s_c : a.c);
    }

    // the block's place in its row-major param (only for the row-major forms)
    int rows = 0, cols = 0;
    int64_t ld = 0, off = 0;
    int param = 0;
    if (GRAD_ROWS || CODES_ROWS) {
        const fp8z1_block blk = a.lut[a.b0 + blockIdx.x];
        rows = blk.rows_real;
        cols = blk.cols_real;
        ld = blk.ld;
        off = blk.src_offset;
        param = blk.param;
    }
    const float* gtile = nullptr;
    bool gvec = false;
    if (GRAD_ROWS) {
        const float* base = a.grad_params[param];
        if (base == nullptr || (reinterpret_cast<uintptr_t>(base) & 3) != 0) {
            if (tid == 0) atomicOr(a.status, FP8Z1_DEV_BADPTR);
            return;  // uniform: the block is left untouched
        }
        gtile = base + off;
        gvec = ((ld & 3) == 0) && ((reinterpret_cast<uintptr_t>(gtile) & 15) == 0);
    }
    uint8_t* ctile = nullptr;
    bool cvec = false;
    if (CODES_ROWS) {
        uint8_t* base = a.code_params[param];
        if (base == nullptr) {
            if (tid == 0) atomicOr(a.status, FP8Z1_DEV_BADPTR);
            return;
        }
        ctile = base + off;
        cvec = ((ld & 3) == 0) && ((reinterpret_cast<uintptr_t>(ctile) & 3) == 0);
    }
    __syncthreads();
    const float gs = s_gscale;
    const StepScalars& c = DEVSC ? s_c : a.c;

    const int64_t base = (int64_t)blockIdx.x * (FP8Z1_BLOCK_ELEMS / 4) + tid;
    float pn[4 * kVec];
    float amax = 0.0f;
#pragma unroll
    for (int j = 0; j < kVec; ++j) {
        const int64_t i = base + j * kThreads;
        float4 g4;
        if (GRAD_ROWS) {
            const int ci = tid + j * kThreads;  // chunk index inside the block
            g4 = load_grad_rows(gtile, ld, ci >> 5, (ci & 31) << 2, rows, cols, gvec);
        } else {
            g4 = __ldcs(a.grad + i);
        }
        float4 p4 = a.master[i];
        float4 m4 = a.mom1[i];
        float4 v4 = a.mom2[i];
        adamw(gs, c, g4.x, p4.x, m4.x, v4.x);
        adamw(gs, c, g4.y, p4.y, m4.y, v4.y);
        adamw(gs, c, g4.z, p4.z, m4.z, v4.z);
        adamw(gs, c, g4.w, p4.w, m4.w, v4.w);
        __stcs(a.mom1 + i, m4);
        __stcs(a.mom2 + i, v4);
        __stcs(a.master + i, p4);
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
    if (tid == 0) a.scales[blockIdx.x] = scale;

    float pd = 0.0f, pp = 0.0f, dd = 0.0f;
    uint32_t under = 0u;
#pragma unroll
    for (int j = 0; j < kVec; ++j) {
        const uint32_t lo = e4m3x2(__fdiv_rn(pn[4 * j + 0], scale), __fdiv_rn(pn[4 * j + 1], scale));
        const uint32_t hi = e4m3x2(__fdiv_rn(pn[4 * j + 2], scale), __fdiv_rn(pn[4 * j + 3], scale));
        const uint32_t q = lo | (hi << 16);
        if (CODES_FOLDED) __stcs(a.codes + base + j * kThreads, q);
        if (CODES_ROWS) {
            const int ci = tid + j * kThreads;
            store_codes_rows(ctile, ld, ci >> 5, (ci & 31) << 2, rows, cols, cvec, q);
        }
        if (MON) {
            const float2 d01 = e4m3x2_decode(lo), d23 = e4m3x2_decode(hi);
            monitor_add(pn[4 * j + 0], d01.x, scale, pd, pp, dd, under);
            monitor_add(pn[4 * j + 1], d01.y, scale, pd, pp, dd, under);
            monitor_add(pn[4 * j + 2], d23.x, scale, pd, pp, dd, under);
            monitor_add(pn[4 * j + 3], d23.y, scale, pd, pp, dd, under);
        }
    }
    if (MON) {
        __shared__ float s_mon[3][kWarps];
        __shared__ uint32_t s_under[kWarps];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            pd += __shfl_xor_sync(0xffffffffu, pd, o);
            pp += __shfl_xor_sync(0xffffffffu, pp, o);
            dd += __shfl_xor_sync(0xffffffffu, dd, o);
            under += __shfl_xor_sync(0xffffffffu, under, o);
        }
        if ((tid & 31) == 0) {
            s_mon[0][tid >> 5] = pd;
            s_mon[1][tid >> 5] = pp;
            s_mon[2][tid >> 5] = dd;
            s_under[tid >> 5] = under;
        }
        __syncthreads();
        if (tid == 0) {
            double tpd = 0.0, tpp = 0.0, tdd = 0.0;
            uint32_t tu = 0u;
            for (int w = 0; w < kWarps; ++w) {
                tpd += s_mon[0][w];
                tpp += s_mon[1][w];
                tdd += s_mon[2][w];
                tu += s_under[w];
            }
            float cosv;
            if (tpp == 0.0 && tdd == 0.0)
                cosv = 1.0f;
            else if (tpp == 0.0 || tdd == 0.0)
                cosv = 0.0f;
            else
                cosv = (float)(tpd / sqrt(tpp * tdd));
            a.block_cos[blockIdx.x] = cosv;
            a.block_underflow[blockIdx.x] = tu;
        }
    }
}

// `hp` may be null (scalars in device memory); when given it must be in domain
int check_common(const fp8z1_layout* L, const fp8z1_adamw_hp* hp, const float* master, const float* m,
                 const float* v, const float* scales, int64_t b0, int64_t b1, const double* d_sumsq,
                 const int32_t* d_found_inf)
{
    if (!master || !m || !v || !scales || !d_sumsq || !d_found_inf || (hp && !in_domain(hp)))
        return FP8Z1_EINVAL;
    const int st = fp8z1::check_range(L, b0, b1);
    if (st != FP8Z1_OK) return st;
    if (b1 - b0 > 0x7fffffffLL) return FP8Z1_EINVAL;
    if (!fp8z1::aligned(master, 16) || !fp8z1::aligned(m, 16) || !fp8z1::aligned(v, 16) ||
        !fp8z1::aligned(scales, 4) || !fp8z1::aligned(d_sumsq, 8) || !fp8z1::aligned(d_found_inf, 4))
        return FP8Z1_EALIGN;
    return FP8Z1_OK;
}

template <bool GR, bool CR, bool CF, bool MON, bool DEVSC>
void launch(const StepArgs& a, int64_t nb, cudaStream_t s)
{
    step_kernel<GR, CR, CF, MON, DEVSC><<<(unsigned)nb, kThreads, 0, s>>>(a);
}

template <bool GR, bool CR, bool CF>
void launch_mon(const StepArgs& a, int64_t nb, cudaStream_t s, bool mon)
{
    const bool dev = a.dsc != nullptr;
    if (mon)
        dev ? launch<GR, CR, CF, true, true>(a, nb, s) : launch<GR, CR, CF, true, false>(a, nb, s);
    else
        dev ? launch<GR, CR, CF, false, true>(a, nb, s) : launch<GR, CR, CF, false, false>(a, nb, s);
}

}  // namespace

extern "C" int fp8z1_step(const fp8z1_layout* L, const fp8z1_adamw_hp* hp, const float* grad_shard,
                          float* master_shard, float* m_shard, float* v_shard, uint8_t* fp8_shard,
                          float* scale_shard, int64_t b0, int64_t b1, const double* d_sumsq,
                          const int32_t* d_found_inf, void* stream)
{
    fp8z1::NvtxRange nvtx_range("fp8z1_step");
    if (!hp) return FP8Z1_EINVAL;
    int st = check_common(L, hp, master_shard, m_shard, v_shard, scale_shard, b0, b1, d_sumsq, d_found_inf);
    if (st != FP8Z1_OK) return st;
    if (!grad_shard || !fp8_shard) return FP8Z1_EINVAL;
    if (!fp8z1::aligned(grad_shard, 16) || !fp8z1::aligned(fp8_shard, 16)) return FP8Z1_EALIGN;
    if (b0 == b1) return FP8Z1_OK;
    StepArgs a = {};
    a.grad = reinterpret_cast<const float4*>(grad_shard);
    a.master = reinterpret_cast<float4*>(master_shard);
    a.mom1 = reinterpret_cast<float4*>(m_shard);
    a.mom2 = reinterpret_cast<float4*>(v_shard);
    a.codes = reinterpret_cast<uint32_t*>(fp8_shard);
    a.scales = scale_shard;
    a.sumsq = d_sumsq;
    a.found_inf = d_found_inf;
    a.lut = L->d_lut;
    a.b0 = b0;
    a.status = L->d_status;
    a.c = scalars(hp);
    launch<false, false, true, false, false>(a, b1 - b0, static_cast<cudaStream_t>(stream));
    return fp8z1::launch_status();
}

namespace {

int step_fused_impl(const fp8z1_layout* L, const fp8z1_adamw_hp* hp, const StepScalars* h_scalars,
                    StepScalars* d_scalars,
                    const float* grad_shard, const float* const* d_grad_params, float* master_shard,
                    float* m_shard, float* v_shard, uint8_t* fp8_shard, uint8_t* const* d_fp8_params,
                    float* scale_shard, float* block_cos, uint32_t* block_underflow, int64_t b0, int64_t b1,
                    const double* d_sumsq, const int32_t* d_found_inf, void* stream)
{
    // exactly one scalar source: hp by value, or d_scalars
    if ((hp == nullptr) == (d_scalars == nullptr)) return FP8Z1_EINVAL;
    int st = check_common(L, hp, master_shard, m_shard, v_shard, scale_shard, b0, b1, d_sumsq, d_found_inf);
    if (st != FP8Z1_OK) return st;
    if (d_scalars && !fp8z1::aligned(d_scalars, 4)) return FP8Z1_EALIGN;
    // exactly one grad source, at least one code destination
    if ((grad_shard == nullptr) == (d_grad_params == nullptr)) return FP8Z1_EINVAL;
    if (fp8_shard == nullptr && d_fp8_params == nullptr) return FP8Z1_EINVAL;
    if ((block_cos == nullptr) != (block_underflow == nullptr)) return FP8Z1_EINVAL;
    if ((block_cos && !fp8z1::aligned(block_cos, 4)) || (block_underflow && !fp8z1::aligned(block_underflow, 4)))
        return FP8Z1_EALIGN;
    if ((grad_shard && !fp8z1::aligned(grad_shard, 16)) || (fp8_shard && !fp8z1::aligned(fp8_shard, 16)) ||
        (d_grad_params && !fp8z1::aligned(d_grad_params, sizeof(void*))) ||
        (d_fp8_params && !fp8z1::aligned(d_fp8_params, sizeof(void*))))
        return FP8Z1_EALIGN;
    if (b0 == b1) return FP8Z1_OK;
    StepArgs a = {};
    a.grad = reinterpret_cast<const float4*>(grad_shard);
    a.master = reinterpret_cast<float4*>(master_shard);
    a.mom1 = reinterpret_cast<float4*>(m_shard);
    a.mom2 = reinterpret_cast<float4*>(v_shard);
    a.codes = reinterpret_cast<uint32_t*>(fp8_shard);
    a.scales = scale_shard;
    a.sumsq = d_sumsq;
    a.found_inf = d_found_inf;
    a.lut = L->d_lut;
    a.b0 = b0;
    a.grad_params = d_grad_params;
    a.code_params = d_fp8_params;
    a.block_cos = block_cos;
    a.block_underflow = block_underflow;
    a.status = L->d_status;
    a.dsc = d_scalars;
    if (hp) a.c = scalars(hp);
    const int64_t nb = b1 - b0;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (h_scalars && cudaMemcpyAsync(d_scalars, h_scalars, sizeof(StepScalars),
                                     cudaMemcpyHostToDevice, s) != cudaSuccess) {
        cudaGetLastError();
        return FP8Z1_ECUDA;
    }
    const bool gr = d_grad_params != nullptr, cr = d_fp8_params != nullptr, cf = fp8_shard != nullptr;
    const bool mon = block_cos != nullptr;
    if (gr) {
        if (cr && cf) launch_mon<true, true, true>(a, nb, s, mon);
        else if (cr) launch_mon<true, true, false>(a, nb, s, mon);
        else launch_mon<true, false, true>(a, nb, s, mon);
    } else {
        if (cr && cf) launch_mon<false, true, true>(a, nb, s, mon);
        else if (cr) launch_mon<false, true, false>(a, nb, s, mon);
        else launch_mon<false, false, true>(a, nb, s, mon);
    }
    return fp8z1::launch_status();
}

}  // namespace

extern "C" int fp8z1_step_fused(const fp8z1_layout* L, const fp8z1_adamw_hp* hp, const float* grad_shard,
                                const float* const* d_grad_params, float* master_shard, float* m_shard,
                                float* v_shard, uint8_t* fp8_shard, uint8_t* const* d_fp8_params,
                                float* scale_shard, float* block_cos, uint32_t* block_underflow,
                                int64_t b0, int64_t b1, const double* d_sumsq,
                                const int32_t* d_found_inf, void* stream)
{
    fp8z1::NvtxRange nvtx_range("fp8z1_step_fused");
    if (!hp) return FP8Z1_EINVAL;
    return step_fused_impl(L, hp, nullptr, nullptr, grad_shard, d_grad_params, master_shard, m_shard, v_shard,
                           fp8_shard, d_fp8_params, scale_shard, block_cos, block_underflow, b0, b1, d_sumsq,
                           d_found_inf, stream);
}

extern "C" int fp8z1_step_fused_dev(const fp8z1_layout* L, const fp8z1_step_scalars* h_scalars,
                                    fp8z1_step_scalars* d_scalars, const float* grad_shard,
                                    const float* const* d_grad_params, float* master_shard, float* m_shard,
                                    float* v_shard, uint8_t* fp8_shard, uint8_t* const* d_fp8_params,
                                    float* scale_shard, float* block_cos, uint32_t* block_underflow, int64_t b0,
                                    int64_t b1, const double* d_sumsq, const int32_t* d_found_inf, void* stream)
{
    fp8z1::NvtxRange nvtx_range("fp8z1_step_fused_dev");
    if (!d_scalars) return FP8Z1_EINVAL;
    return step_fused_impl(L, nullptr, h_scalars, d_scalars, grad_shard, d_grad_params, master_shard, m_shard,
                           v_shard, fp8_shard, d_fp8_params, scale_shard, block_cos, block_underflow, b0, b1,
                           d_sumsq, d_found_inf, stream);
}

extern "C" int fp8z1_step_scalars_from_hp(const fp8z1_adamw_hp* hp, fp8z1_step_scalars* out)
{
    if (!hp || !out || !in_domain(hp)) return FP8Z1_EINVAL;
    *out = scalars(hp);
    return FP8Z1_OK;
}
