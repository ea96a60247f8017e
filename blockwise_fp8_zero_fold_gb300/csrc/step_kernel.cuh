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
// One CTA of 512 threads per block of 16384 elements, three CTAs per SM;
// thread t owns the float4 chunks t, t+512, ..., t+3584 of the block (chunk i
// is row i/32, columns 4*(i%32) .. +3 of the 128x128 block, so a warp covers
// one block row).  A partial block whose real columns fit in 64, 32, ... (W
// float4 chunks a row, a power of two) has each warp cover 32 / W rows at a
// time instead, so its warps finish in fewer passes (ragged's step 2.405 ->
// 2.313 ms); the new master of chunk j of thread t still waits in shared-memory
// slot t + 512 j.  It streams grad / master / m / v in, updates them, writes
// master / m / v back at once and keeps its 32 new master values in its slots
// of a 64 KB shared array while the CTA reduces the block amax (warp
// shuffles, then 16 partials in shared memory).  The codes are then produced
// from shared memory: no second pass over HBM.
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
//
// Padding: the elements of a block outside its real rows and columns are zero
// in grad, master, m and v (fold writes them so), and the update maps them to
// zero again (g = 0 gives m = v = +0 and p = fma(-a, +0, +0) = +0), so a block
// that is not a full 128x128 tile skips the float4 chunks that hold padding
// only: no load, no store, new master 0 (which leaves the amax alone), and no
// code to compute -- 0x00 goes to a folded code shard, nothing to the
// row-major params.  (Computing those codes anyway, four divisions a chunk,
// cost the ragged workload's step 4-5%.)  Full tiles take the loops without
// the test.
//
// Row-major grads and codes of a param whose C is not a multiple of 4 start
// each row at a different alignment; a chunk there is read and written with
// the widest access its address allows (16 or 8 bytes of grads, 4 or 2 of
// codes), one element at a time only where it must be.  Those grads are read
// through L1 (the read-only path; nothing writes them during the step), so
// the four single-element loads of a warp fetch their lines from L2 once:
// streaming loads, which L1 does not keep, fetched them four times (ragged's
// step 2.314 -> 2.277 ms).
#pragma once

#include <math.h>

#include <atomic>

#include "checked.cuh"
#include "step_args.h"

namespace fp8z1 {
namespace stepk {

__device__ __forceinline__ float warp_max(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// The 4 grads of chunk (r, c) of a row-major tile; zeros outside the real
// extent.  first: the element index of tile[0] in its param, elems: the
// param's extent (a checked build tests each access against them).
__device__ __forceinline__ float4 load_grad_rows(const float* tile, int64_t ld, int r, int c, int rows,
                                                 int cols, bool vec, int64_t first, int64_t elems)
{
    float4 g = make_float4(0.f, 0.f, 0.f, 0.f);
    if (r < rows) {
        const int64_t at = first + r * ld + c;
        const float* src = tile + r * ld + c;
        if (vec) {  // ld % 4 == 0: a 4-column group is all real or all padding
            if (c < cols && in_extent(at, 4, elems)) g = __ldcs(reinterpret_cast<const float4*>(src));
        } else {
            // rows of a param whose C % 4 != 0 start at different alignments:
            // the widest access this chunk's address allows, when it is all
            // real, through L1
            const uintptr_t ad = reinterpret_cast<uintptr_t>(src);
            if (c + 3 < cols && (ad & 15) == 0) {
                if (in_extent(at, 4, elems)) g = __ldg(reinterpret_cast<const float4*>(src));
            } else if (c + 3 < cols && (ad & 7) == 0) {
                if (in_extent(at, 4, elems)) {
                    const float2 lo = __ldg(reinterpret_cast<const float2*>(src));
                    const float2 hi = __ldg(reinterpret_cast<const float2*>(src + 2));
                    g = make_float4(lo.x, lo.y, hi.x, hi.y);
                }
            } else {
                if (c + 0 < cols && in_extent(at + 0, 1, elems)) g.x = __ldg(src + 0);
                if (c + 1 < cols && in_extent(at + 1, 1, elems)) g.y = __ldg(src + 1);
                if (c + 2 < cols && in_extent(at + 2, 1, elems)) g.z = __ldg(src + 2);
                if (c + 3 < cols && in_extent(at + 3, 1, elems)) g.w = __ldg(src + 3);
            }
        }
    }
    return g;
}

__device__ __forceinline__ void store_codes_rows(uint8_t* tile, int64_t ld, int r, int c, int rows,
                                                 int cols, bool vec, uint32_t q, int64_t first, int64_t elems)
{
    if (r >= rows) return;
    const int64_t at = first + r * ld + c;
    uint8_t* dst = tile + r * ld + c;
    if (vec) {
        if (c < cols && in_extent(at, 4, elems)) __stcs(reinterpret_cast<unsigned int*>(dst), q);
    } else {
        const uintptr_t ad = reinterpret_cast<uintptr_t>(dst);
        if (c + 3 < cols && (ad & 3) == 0) {
            if (in_extent(at, 4, elems)) __stcs(reinterpret_cast<unsigned int*>(dst), q);
        } else if (c + 3 < cols && (ad & 1) == 0) {
            if (in_extent(at, 4, elems)) {
                __stcs(reinterpret_cast<unsigned short*>(dst), (unsigned short)(q & 0xffffu));
                __stcs(reinterpret_cast<unsigned short*>(dst + 2), (unsigned short)(q >> 16));
            }
        } else {
#pragma unroll
            for (int b = 0; b < 4; ++b)
                if (c + b < cols && in_extent(at + b, 1, elems)) dst[b] = (uint8_t)(q >> (8 * b));
        }
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

// Dynamic shared memory of the kernel: the block's 16384 new masters, which
// each thread writes to its own slots (chunk j of thread t at t + 512 j) and
// reads back after the block-amax barrier.  Keeping them there rather than in
// registers lets three CTAs fit per SM (40 registers) instead of two (64):
// MoE's full-tile step 6.010 -> 5.894 ms, ragged's padding-aware one 2.806 ->
// 2.505 ms.  The forms with the quantisation monitors keep two CTAs per SM
// (up to 64 registers): squeezed to 40 with three, their extra sums ran 9%
// slower on MoE (7.37 against 6.78 ms).
constexpr int kMasterSmemBytes = kThreads * kVec * 16;

// Where this thread's chunks of a block sit.  A warp takes 32 / W rows at a
// time, W = the block's real chunks a row rounded up to a power of two (sh =
// log2(32 / W); sh = 0 for a block with more than 64 real columns and in
// every full-tile launch): lane l has chunk l % W of row l / W of the warp's
// rows, and chunk j of thread t is row rbase + j * (16 << sh), folded float4
// index ibase + j * (512 << sh); jn of them hold real elements.
struct ChunkPlace {
    int64_t ibase;
    int rbase, col, sh, jn;
};

template <bool PAD>
__device__ __forceinline__ ChunkPlace chunk_place(int64_t kb, int tid, int rows, int cols, int sh)
{
    ChunkPlace c;
    const int lane = tid & 31, warp = tid >> 5;
    const int rsub = lane >> (5 - sh), cc = lane & ((32 >> sh) - 1);
    c.sh = sh;
    c.rbase = (warp << sh) + rsub;
    c.col = cc << 2;
    c.ibase = kb * (FP8Z1_BLOCK_ELEMS / 4) + (int64_t)c.rbase * (FP8Z1_TILE / 4) + cc;
    c.jn = kVec;
    if (PAD) {
        // tasks of 2^sh rows this lane has real rows in, then the chunks j < jn
        const int tasks = rows > rsub ? (rows - rsub + (1 << sh) - 1) >> sh : 0;
        c.jn = c.col >= cols ? 0 : min(kVec, max(0, (tasks - warp + 15) >> 4));
    }
    return c;
}

// The update of this thread's 8 float4 chunks of the block (placed by cp):
// new masters into pn[j * kThreads] (shared memory), their largest magnitude
// into amax.  PAD: the chunks j >= cp.jn hold padding only and are skipped.
template <bool GRAD_ROWS, bool PAD>
__device__ __forceinline__ void update_chunks(const StepArgs& a, const StepScalars& c, float gs, const ChunkPlace& cp,
                                              const float* gtile, int64_t ld, int rows, int cols,
                                              bool gvec, int64_t first, int64_t elems, float4* pn,
                                              float& amax)
{
#pragma unroll
    for (int j = 0; j < kVec; ++j) {
        if (PAD && j >= cp.jn) {
            pn[j * kThreads] = make_float4(0.f, 0.f, 0.f, 0.f);
            continue;
        }
        const int64_t i = cp.ibase + ((int64_t)j * kThreads << (PAD ? cp.sh : 0));
        const int row = cp.rbase + ((16 * j) << (PAD ? cp.sh : 0));
        float4 g4;
        if (GRAD_ROWS) {
            if (!PAD && gvec) {  // a full tile (every launch without PAD), 16-byte rows
                const int64_t at = (int64_t)row * ld + cp.col;
                g4 = in_extent(first + at, 4, elems) ? __ldcs(reinterpret_cast<const float4*>(gtile + at))
                                                     : make_float4(0.f, 0.f, 0.f, 0.f);
            } else {
                g4 = load_grad_rows(gtile, ld, row, cp.col, rows, cols, gvec, first, elems);
            }
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
        pn[j * kThreads] = p4;
        amax = fmaxf(amax, fmaxf(fmaxf(fabsf(p4.x), fabsf(p4.y)), fmaxf(fabsf(p4.z), fabsf(p4.w))));
    }
}

template <bool GRAD_ROWS, bool CODES_ROWS, bool CODES_FOLDED, bool MON, int SC, bool PAD>
__global__ void __launch_bounds__(kThreads, MON ? 2 : 3) step_kernel(const StepArgs a)
{
    if (*a.found_inf != 0) return;  // skipped step: write nothing
    // Where the update reads its scalars: shared memory for the scalars from
    // device memory, and for the by-value full-tile forms that read the grads
    // row-major -- at 40 registers those spilled reading the parameters at
    // every use (MoE: 6.010 -> 5.907 ms from shared memory); the kernel
    // parameters for the rest, whose issue-bound padding-aware and folded
    // forms ran up to 9% slower with the extra shared-memory loads.  The select
    // form keeps its two sets as parameters behind one uniform branch.
    constexpr bool kSmemScalars = SC == kScDevice || (SC != kScSelect && GRAD_ROWS && !PAD);
    __shared__ float s_gscale;
    __shared__ float s_amax[kWarps];
    __shared__ StepScalars s_c;
    __shared__ int s_alt;
    const int tid = threadIdx.x;
    if (tid == 0) {
        if (kSmemScalars) s_c = SC == kScDevice ? *a.dsc : a.c;
        const bool alt = SC == kScSelect && *a.select != 0;
        s_alt = alt;
        s_gscale = grad_factor(*a.sumsq, kSmemScalars ? s_c : (alt ? a.c2 : a.c));
    }

    // the block's place in its row-major param and its real extent
    const int64_t kb = a.blk_off + blockIdx.x;  // block index from b0
    int rows = FP8Z1_TILE, cols = FP8Z1_TILE;
    int64_t ld = 0, off = 0;
    int param = 0;
    int64_t elems = 0;  // the param's extent (checked builds)
    if (GRAD_ROWS || CODES_ROWS || PAD) {
        const fp8z1_block blk = a.lut[a.b0 + kb];
        rows = blk.rows_real;
        cols = blk.cols_real;
        ld = blk.ld;
        off = blk.src_offset;
        param = blk.param;
#if FP8Z1_CHECKED
        if (GRAD_ROWS || CODES_ROWS) elems = a.param_elems[param];
#endif
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

    const int64_t base = kb * (FP8Z1_BLOCK_ELEMS / 4) + tid;
    // narrow blocks take several rows a warp, except into a folded code shard
    // (which wants every chunk of the block written)
    int sh = 0;
    if (PAD && !CODES_FOLDED) {
        const int nc = (cols + 3) >> 2;
        sh = nc > 16 ? 0 : nc > 8 ? 1 : nc > 4 ? 2 : nc > 2 ? 3 : nc > 1 ? 4 : 5;
    }
    const ChunkPlace cp = chunk_place<PAD>(kb, tid, rows, cols, sh);
    extern __shared__ float4 s_pn[];  // kMasterSmemBytes: the block's new masters
    float4* const pn = s_pn + tid;
    float amax = 0.0f;
    if constexpr (SC == kScSelect) {
        // one uniform branch, each side with its scalars as kernel-parameter
        // operands (no registers held for them)
        if (s_alt)
            update_chunks<GRAD_ROWS, PAD>(a, a.c2, gs, cp, gtile, ld, rows, cols, gvec, off, elems, pn,
                                          amax);
        else
            update_chunks<GRAD_ROWS, PAD>(a, a.c, gs, cp, gtile, ld, rows, cols, gvec, off, elems, pn,
                                          amax);
    } else {
        update_chunks<GRAD_ROWS, PAD>(a, kSmemScalars ? s_c : a.c, gs, cp, gtile, ld, rows, cols,
                                      gvec, off, elems, pn, amax);
    }

    amax = warp_max(amax);
    if ((tid & 31) == 0) s_amax[tid >> 5] = amax;
    __syncthreads();
    float bmax = s_amax[0];
#pragma unroll
    for (int w = 1; w < kWarps; ++w) bmax = fmaxf(bmax, s_amax[w]);
    const float scale = bmax == 0.0f ? 1.0f : __fdiv_rn(bmax, 448.0f);
    if (tid == 0) a.scales[kb] = scale;

    float pd = 0.0f, pp = 0.0f, dd = 0.0f;
    uint32_t under = 0u;
    // chunks j >= jn hold padding only: their new masters are 0, their codes
    // 0x00 (stored only into a folded code shard), their monitor terms 0
#pragma unroll
    for (int j = 0; j < kVec; ++j) {
        if (PAD && j >= cp.jn) {
            if (CODES_FOLDED) __stcs(a.codes + base + j * kThreads, 0u);
            continue;
        }
        const float4 p = pn[j * kThreads];
        const uint32_t lo = e4m3x2(__fdiv_rn(p.x, scale), __fdiv_rn(p.y, scale));
        const uint32_t hi = e4m3x2(__fdiv_rn(p.z, scale), __fdiv_rn(p.w, scale));
        const uint32_t q = lo | (hi << 16);
        if (CODES_FOLDED) __stcs(a.codes + base + j * kThreads, q);
        if (CODES_ROWS) {
            const int row = cp.rbase + ((16 * j) << (PAD ? cp.sh : 0));
            if (!PAD && cvec) {  // a full tile, 4-byte aligned rows
                const int64_t at = (int64_t)row * ld + cp.col;
                if (in_extent(off + at, 4, elems)) __stcs(reinterpret_cast<unsigned int*>(ctile + at), q);
            } else {
                store_codes_rows(ctile, ld, row, cp.col, rows, cols, cvec, q, off, elems);
            }
        }
        if (MON) {
            const float2 d01 = e4m3x2_decode(lo), d23 = e4m3x2_decode(hi);
            monitor_add(p.x, d01.x, scale, pd, pp, dd, under);
            monitor_add(p.y, d01.y, scale, pd, pp, dd, under);
            monitor_add(p.z, d23.x, scale, pd, pp, dd, under);
            monitor_add(p.w, d23.y, scale, pd, pp, dd, under);
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
            a.block_cos[kb] = cosv;
            a.block_underflow[kb] = tu;
        }
    }
}

// `hp` may be null (scalars in device memory); when given it must be in domain

// Lets `kernel` take kMasterSmemBytes of dynamic shared memory on the current
// device (an attribute set per device), once per device; a failure shows as
// the launch's error.
inline void allow_master_smem(const void* kernel, std::atomic<uint64_t>& set)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return;
    }
    const uint64_t bit = dev < 64 ? (1ull << dev) : 0ull;
    if (bit && (set.load(std::memory_order_relaxed) & bit)) return;
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kMasterSmemBytes) ==
        cudaSuccess)
        set.fetch_or(bit, std::memory_order_relaxed);
    else
        cudaGetLastError();
}

template <bool PAD>
void launch(const StepArgs& a, int64_t nb, cudaStream_t s, unsigned forms)
{
    // the forms the entry points use: grads folded or row-major, codes to
    // the folded shard and/or row-major, with or without monitors, scalars by
    // value, in device memory, or two sets by value picked by a device flag
    // (without monitors)
#define FP8Z1_STEP_FORM(GR, CR, CF, MON, SCAL)                                                       \
    if (forms == ((GR ? kGradRows : 0u) | (CR ? kCodesRows : 0u) | (CF ? kCodesFolded : 0u) |         \
                  (MON ? kMonitors : 0u) | (SCAL == kScDevice ? kDevScalars : 0u) |                   \
                  (SCAL == kScSelect ? kSelScalars : 0u))) {                                          \
        static std::atomic<uint64_t> smem_set{0}; /* devices whose attribute is set */                  \
        allow_master_smem(reinterpret_cast<const void*>(&step_kernel<GR, CR, CF, MON, SCAL, PAD>), smem_set); \
        step_kernel<GR, CR, CF, MON, SCAL, PAD><<<(unsigned)nb, kThreads, kMasterSmemBytes, s>>>(a);  \
        return;                                                                                      \
    }
#define FP8Z1_STEP_FORMS_GC(GR, CR, CF)                                                              \
    FP8Z1_STEP_FORM(GR, CR, CF, false, kScValue)                                                     \
    FP8Z1_STEP_FORM(GR, CR, CF, false, kScDevice)                                                    \
    FP8Z1_STEP_FORM(GR, CR, CF, true, kScValue)                                                      \
    FP8Z1_STEP_FORM(GR, CR, CF, true, kScDevice)                                                     \
    FP8Z1_STEP_FORM(GR, CR, CF, false, kScSelect)
    FP8Z1_STEP_FORMS_GC(true, true, true)
    FP8Z1_STEP_FORMS_GC(true, true, false)
    FP8Z1_STEP_FORMS_GC(true, false, true)
    FP8Z1_STEP_FORMS_GC(false, true, true)
    FP8Z1_STEP_FORMS_GC(false, true, false)
    FP8Z1_STEP_FORMS_GC(false, false, true)
#undef FP8Z1_STEP_FORMS_GC
#undef FP8Z1_STEP_FORM
}

template <bool PAD>
bool is_value_kernel(const void* func)
{
#define FP8Z1_STEP_VALUE_FORM(GR, CR, CF, MON) \
    if (func == reinterpret_cast<const void*>(&step_kernel<GR, CR, CF, MON, kScValue, PAD>)) return true;
#define FP8Z1_STEP_VALUE_FORMS(GR, CR, CF) FP8Z1_STEP_VALUE_FORM(GR, CR, CF, false) FP8Z1_STEP_VALUE_FORM(GR, CR, CF, true)
    FP8Z1_STEP_VALUE_FORMS(true, true, true)
    FP8Z1_STEP_VALUE_FORMS(true, true, false)
    FP8Z1_STEP_VALUE_FORMS(true, false, true)
    FP8Z1_STEP_VALUE_FORMS(false, true, true)
    FP8Z1_STEP_VALUE_FORMS(false, true, false)
    FP8Z1_STEP_VALUE_FORMS(false, false, true)
#undef FP8Z1_STEP_VALUE_FORMS
#undef FP8Z1_STEP_VALUE_FORM
    return false;
}

}  // namespace stepk
}  // namespace fp8z1
