// Global grad norm: the sum of squares of the loss-scaled FP32 grads of a
// block range, plus the inf/nan flag -- read from the folded grad shard
// (fp8z1_grad_norm) or straight from the row-major grads through the block
// lookup table, optionally storing the folded blocks on the way
// (fp8z1_fold_norm: the fold of the grads fused with the norm).
//
// "DeepSpeed ZeRO 优化" §七 梯度裁剪: the global norm is the square root of the
// sum over every rank of its partial sum of squares (an all-reduce); the clip
// coefficient is formed from it.  §六 / §九 Q6: an inf or nan among the grads
// skips the step.  "面向 Blockwise FP8 量化的 ZeRO 优化器设计" §总结 /
// §参数布局变换: the reduced grads are folded into the optimizer's layout.
//
// Accuracy: each square is split exactly into float hi + lo parts
// (x*x and fma(x, x, -x*x)), and a thread adds its 32 squares of a unit (half
// a block, below) with error-free sums -- in two interleaved chains of 16,
// each step a Fast2Sum of the larger and the smaller of the running sum and
// the new square (both non-negative), the two chains joined by one more -- so
// its per-unit partial is within about 32^2 ulp^2 of the exact value;
// partials are then summed in double.  The result is well inside 1e-12
// relative of the exact sum -- close enough that the clip coefficient formed
// from it rounds to the same FP32 number as one formed from the exact sum,
// except in rare ties.  The float path is exact enough only while the partial
// stays in [2^-90, 2^100), or is 0 because every value is 0: an inf or nan, a
// square that overflows, or tiny values (whose squares underflow, possibly to
// a partial of 0) land outside, and then the thread redoes those 32 values in
// double, where the square of any float is exact.
//
// Latency: the unit of work is half a block (8192 values; read row-major, 64
// rows of a block).  Three persistent CTAs of 256 threads per SM each walk a
// contiguous run of units; each thread loads the next unit's 32 values (and,
// reading row-major, looks up the block after that in the table) while it sums
// the current ones, so an SM always has three units' worth of loads in flight.
// A pure read of this shape reaches about 7.5 TB/s on a GB300; one CTA of 512
// threads per SM holding whole blocks reached about 6.4.
//
// Reduction: each CTA writes one double to a workspace, and the last CTA to
// finish (an atomic ticket, no waiting) adds the partials in a fixed order.
// The result is deterministic for a given device and range.
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>

#include "checked.cuh"

namespace {

constexpr int kThreads = 256;
constexpr int kCtasPerSm = 3;
constexpr int kVec = 8;                                           // float4 per thread and unit
constexpr int kUnitElems = kThreads * kVec * 4;                   // 8192: half a block
constexpr int kUnitsPerBlock = FP8Z1_BLOCK_ELEMS / kUnitElems;    // 2
constexpr int kUnitRows = FP8Z1_TILE / kUnitsPerBlock;            // 64 rows of a block
constexpr int kWarps = kThreads / 32;
static_assert(kUnitsPerBlock * kUnitElems == FP8Z1_BLOCK_ELEMS, "a block is a whole number of units");
static_assert(kUnitRows * FP8Z1_TILE == kUnitElems, "a unit is whole rows of a block");

// a + b = s + err exactly, for a, b >= 0 (Dekker's Fast2Sum on max, min).
// An inf gives s = inf; a nan is dropped by fmaxf / fminf, so the caller
// must see it elsewhere (add_square: in lo).
__device__ __forceinline__ void fast_two_sum(float a, float b, float& s, float& err)
{
    const float big = fmaxf(a, b), small = fminf(a, b);
    s = __fadd_rn(big, small);
    err = __fsub_rn(small, __fsub_rn(s, big));
}

// hi + lo += x*x.  A nan x makes lo nan (e is nan); an inf x makes hi inf.
__device__ __forceinline__ void add_square(float x, float& hi, float& lo)
{
    const float sq = __fmul_rn(x, x);
    const float e = __fmaf_rn(x, x, -sq);  // x*x = sq + e exactly (no under/overflow)
    float t;
    fast_two_sum(hi, sq, hi, t);
    lo = __fadd_rn(lo, __fadd_rn(t, e));
}

// The float partial is exact enough when it lies in [2^-90, 2^100) and lo is
// a number, or when every value was zero (nz == 0).
__device__ __forceinline__ bool float_path_ok(float hi, float lo, unsigned nz)
{
    return hi < 0x1p100f && lo == lo && (hi >= 0x1p-90f || nz == 0u);
}

__device__ __forceinline__ void add_square_exact(float x, double& acc, int& bad)
{
    if ((__float_as_uint(x) & 0x7f800000u) == 0x7f800000u)
        bad = 1;
    else
        acc += (double)x * (double)x;  // exact product of two floats
}

__device__ __forceinline__ double warp_sum(double v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ void sum_unit(const float4 (&x)[kVec], double& acc, int& bad)
{
    float hi0 = 0.0f, lo0 = 0.0f, hi1 = 0.0f, lo1 = 0.0f;
    unsigned bits = 0u;
#pragma unroll
    for (int j = 0; j < kVec; ++j) {
        bits |= __float_as_uint(x[j].x) | __float_as_uint(x[j].y) | __float_as_uint(x[j].z) |
                __float_as_uint(x[j].w);
        add_square(x[j].x, hi0, lo0);
        add_square(x[j].y, hi1, lo1);
        add_square(x[j].z, hi0, lo0);
        add_square(x[j].w, hi1, lo1);
    }
    float hi, t;
    fast_two_sum(hi0, hi1, hi, t);
    const float lo = __fadd_rn(__fadd_rn(lo0, lo1), t);
    const unsigned nz = bits & 0x7fffffffu;  // any nonzero magnitude
    if (float_path_ok(hi, lo, nz)) {
        acc += (double)hi;
        acc += (double)lo;
    } else {
#pragma unroll
        for (int j = 0; j < kVec; ++j) {
            add_square_exact(x[j].x, acc, bad);
            add_square_exact(x[j].y, acc, bad);
            add_square_exact(x[j].z, acc, bad);
            add_square_exact(x[j].w, acc, bad);
        }
    }
}

// Where the grads of one block come from: the folded shard, a block of the
// row-major params (through the block table), a run of at most 16384
// consecutive elements of a param the range holds whole (from the layout's
// run table), or a run of at most 16384 elements of one contiguous span of a
// param (whole row-block strips of a param the range cuts: a strip is 128
// full rows, and consecutive strips are consecutive in memory).  A sum of
// squares needs no block structure, so only partial strips need the table.
// Each of these is two units: its first and second 8192 values (for a block
// of the row-major params, its rows 0-63 and 64-127).
// A flat range of grads (an MXFP8 shard) is read the same way, run by run.
enum Src { kFolded, kRows, kParams, kSpan, kFlat };

// Where unit k's grads live in the row-major params.
struct RowSrc {
    const float* tile;
    int64_t ld;
    int rows, cols;
    int count;  // kParams, kSpan: elements in the run
    bool vec;   // 16-byte loads (kRows: ld % 4 == 0 and an aligned tile; kParams, kSpan: an aligned run)
    bool bad;   // null or misaligned param pointer
#if FP8Z1_CHECKED
    int64_t first;  // element index of tile[0] in its param
    int64_t elems;  // the param's extent
#endif
};

// Whether tile[idx .. idx + w) lies inside its param (checked builds test it).
__device__ __forceinline__ bool src_ok(const RowSrc& s, int64_t idx, int w)
{
#if FP8Z1_CHECKED
    return fp8z1::in_extent(s.first + idx, w, s.elems);
#else
    (void)s;
    (void)idx;
    (void)w;
    return true;
#endif
}

__device__ __forceinline__ RowSrc row_src(const fp8z1_block* __restrict__ lut,
                                          const float* const* __restrict__ params,
                                          const int64_t* __restrict__ param_elems, int64_t k)
{
    const fp8z1_block blk = lut[k];
    const float* base = params[blk.param];
    RowSrc s;
#if FP8Z1_CHECKED
    s.first = blk.src_offset;
    s.elems = param_elems[blk.param];
#else
    (void)param_elems;
#endif
    s.bad = base == nullptr || (reinterpret_cast<uintptr_t>(base) & 3) != 0;
    s.tile = s.bad ? nullptr : base + blk.src_offset;
    s.ld = blk.ld;
    s.rows = blk.rows_real;
    s.cols = blk.cols_real;
    s.vec = !s.bad && (blk.ld & 3) == 0 && (reinterpret_cast<uintptr_t>(s.tile) & 15) == 0;
    return s;
}

__device__ __forceinline__ RowSrc param_src(const fp8z1_unit* __restrict__ units,
                                            const float* const* __restrict__ params,
                                            const int64_t* __restrict__ param_elems, int64_t u)
{
    const fp8z1_unit un = units[u];
    const float* base = params[un.param];
    RowSrc s = {};
#if FP8Z1_CHECKED
    s.first = un.offset;
    s.elems = param_elems[un.param];
#else
    (void)param_elems;
#endif
    s.bad = base == nullptr || (reinterpret_cast<uintptr_t>(base) & 3) != 0;
    s.tile = s.bad ? nullptr : base + un.offset;
    s.count = un.count;
    s.vec = !s.bad && (reinterpret_cast<uintptr_t>(s.tile) & 15) == 0;
    return s;
}

// Run k of a span: elements span_offset + 16384 k .. of param span_param.
__device__ __forceinline__ RowSrc span_src(const float* const* __restrict__ params,
                                           const int64_t* __restrict__ param_elems, int32_t param,
                                           int64_t offset, int64_t elems, int64_t k)
{
    const float* base = params[param];
    RowSrc s = {};
    s.bad = base == nullptr || (reinterpret_cast<uintptr_t>(base) & 3) != 0;
    const int64_t o = k * FP8Z1_BLOCK_ELEMS;
#if FP8Z1_CHECKED
    s.first = offset + o;
    s.elems = param_elems[param];
#else
    (void)param_elems;
#endif
    s.tile = s.bad ? nullptr : base + offset + o;
    s.count = (int)(elems - o < FP8Z1_BLOCK_ELEMS ? elems - o : FP8Z1_BLOCK_ELEMS);
    s.vec = !s.bad && (reinterpret_cast<uintptr_t>(s.tile) & 15) == 0;
    return s;
}

// Run k of a flat range of `elems` grads at `base` (16-byte aligned):
// elements 16384 k .. , the last run possibly short.
__device__ __forceinline__ RowSrc flat_src(const float* base, int64_t elems, int64_t k)
{
    RowSrc s = {};
    const int64_t o = k * FP8Z1_BLOCK_ELEMS;
#if FP8Z1_CHECKED
    s.first = o;
    s.elems = elems;
#endif
    s.tile = base + o;
    s.count = (int)(elems - o < FP8Z1_BLOCK_ELEMS ? elems - o : FP8Z1_BLOCK_ELEMS);
    s.vec = true;
    return s;
}

struct NormArgs {
    const float4* g;              // folded grads at block b0 (kFolded); the flat grads (kFlat)
    const fp8z1_block* lut;       // kRows
    const fp8z1_unit* units;      // kParams
    const float* const* params;   // kRows, kParams, kSpan: row-major FP32 grads
    const int64_t* param_elems;   // kRows, kParams, kSpan: each param's extent (checked builds test against it)
    int64_t span_offset;          // kSpan: first element of the span in its param ...
    int64_t span_elems;           // ... its length ... (kFlat: the flat range's length)
    int32_t span_param;           // ... and the param
    float4* store;                // STORE: folded grads at block b0
    int64_t b0;                   // first block (kRows: LUT index) or run (kParams)
    int64_t nblocks;              // blocks of 16384, the last one possibly partial (2 units each)
    double* partials;             // one per CTA
    unsigned* counter;
    unsigned* status;
    double* sumsq;
    int32_t* found_inf;
};

// Issue the loads of unit u (index from the launch's first block; the block
// is u / 2, h = u % 2 its half): this thread's 32 values.  Chunk j is
// ci = tid + 256 j of the unit: for a block, block row 64 h + ci / 32 and
// columns 4 (ci % 32) .. + 3; for a run of a param, elements
// 8192 h + 4 ci .. + 3.  Zeros outside the real extent.
template <Src SRC>
__device__ __forceinline__ void load_unit(const NormArgs& a, const RowSrc& s, int64_t u, int tid,
                                          float4 (&x)[kVec])
{
    const int h = (int)(u % kUnitsPerBlock);
    if constexpr (SRC == kFolded) {
        const float4* p = a.g + u * (kUnitElems / 4) + tid;
#pragma unroll
        for (int j = 0; j < kVec; ++j) x[j] = __ldcs(p + j * kThreads);
    } else if constexpr (SRC == kParams || SRC == kSpan || SRC == kFlat) {
        const int e0 = h * kUnitElems;
        if (s.vec && s.count == FP8Z1_BLOCK_ELEMS) {  // a whole, aligned run
            const float4* p = reinterpret_cast<const float4*>(s.tile + e0) + tid;
#pragma unroll
            for (int j = 0; j < kVec; ++j)
                x[j] = src_ok(s, e0 + 4 * (tid + j * kThreads), 4) ? __ldcs(p + j * kThreads)
                                                                  : make_float4(0.f, 0.f, 0.f, 0.f);
            return;
        }
#pragma unroll
        for (int j = 0; j < kVec; ++j) {
            const int e = e0 + 4 * (tid + j * kThreads);
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            if (!s.bad && e < s.count) {
                const float* src = s.tile + e;
                if (s.vec && e + 4 <= s.count) {
                    if (src_ok(s, e, 4)) v = __ldcs(reinterpret_cast<const float4*>(src));
                } else {
                    if (src_ok(s, e, 1)) v.x = __ldcs(src + 0);
                    if (e + 1 < s.count && src_ok(s, e + 1, 1)) v.y = __ldcs(src + 1);
                    if (e + 2 < s.count && src_ok(s, e + 2, 1)) v.z = __ldcs(src + 2);
                    if (e + 3 < s.count && src_ok(s, e + 3, 1)) v.w = __ldcs(src + 3);
                }
            }
            x[j] = v;
        }
    } else {
        const int r0 = h * kUnitRows;
        if (s.vec && s.rows == FP8Z1_TILE && s.cols == FP8Z1_TILE) {
            // a full, aligned block: chunk j sits 8 rows below chunk j-1
            const int64_t off = (int64_t)(r0 + (tid >> 5)) * s.ld + ((tid & 31) << 2);
            const float* src = s.tile + off;
            const int64_t step = (kThreads / 32) * s.ld;
#pragma unroll
            for (int j = 0; j < kVec; ++j)
                x[j] = src_ok(s, off + j * step, 4) ? __ldcs(reinterpret_cast<const float4*>(src + j * step))
                                                   : make_float4(0.f, 0.f, 0.f, 0.f);
            return;
        }
#pragma unroll
        for (int j = 0; j < kVec; ++j) {
            const int ci = tid + j * kThreads;
            const int r = r0 + (ci >> 5), c = (ci & 31) << 2;
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            if (!s.bad && r < s.rows) {
                const int64_t off = r * s.ld + c;
                const float* src = s.tile + off;
                if (s.vec) {  // a 4-column group is then all real or all padding
                    if (c < s.cols && src_ok(s, off, 4)) v = __ldcs(reinterpret_cast<const float4*>(src));
                } else {
                    if (c + 0 < s.cols && src_ok(s, off + 0, 1)) v.x = __ldcs(src + 0);
                    if (c + 1 < s.cols && src_ok(s, off + 1, 1)) v.y = __ldcs(src + 1);
                    if (c + 2 < s.cols && src_ok(s, off + 2, 1)) v.z = __ldcs(src + 2);
                    if (c + 3 < s.cols && src_ok(s, off + 3, 1)) v.w = __ldcs(src + 3);
                }
            }
            x[j] = v;
        }
    }
}

// Where unit u's block lives.
template <Src SRC>
__device__ __forceinline__ RowSrc src_of(const NormArgs& a, int64_t u)
{
    const int64_t k = u / kUnitsPerBlock;
    if (SRC == kRows) return row_src(a.lut, a.params, a.param_elems, a.b0 + k);
    if (SRC == kParams) return param_src(a.units, a.params, a.param_elems, a.b0 + k);
    if (SRC == kSpan) return span_src(a.params, a.param_elems, a.span_param, a.span_offset, a.span_elems, k);
    if (SRC == kFlat) return flat_src(reinterpret_cast<const float*>(a.g), a.span_elems, k);
    return RowSrc{};
}

// Sum (and store) unit u, whose values are in x.  Folded, unit u is the
// 8192 consecutive values from 8192 u: chunk ci of it holds elements
// 4 ci .. + 3, which is where load_unit took them from.
template <Src SRC, bool STORE>
__device__ __forceinline__ void finish_unit(const NormArgs& a, const RowSrc& s, int64_t u, int tid,
                                            const float4 (&x)[kVec], double& acc, int& bad)
{
    if (SRC != kFolded && s.bad) {  // unreadable grads: nothing is summed or stored
        if (tid == 0) atomicOr(a.status, FP8Z1_DEV_BADPTR);
        bad = 1;          // raise found_inf so the step is skipped
        return;
    }
    if (STORE) {
        float4* dst = a.store + u * (kUnitElems / 4) + tid;
#pragma unroll
        for (int j = 0; j < kVec; ++j) __stcs(dst + j * kThreads, x[j]);
    }
    sum_unit(x, acc, bad);
}

template <Src SRC, bool STORE>
__global__ void __launch_bounds__(kThreads, kCtasPerSm) norm_kernel(const NormArgs a)
{
    __shared__ double s_part[kWarps];
    __shared__ int s_last;
    const int tid = threadIdx.x;
    const int64_t nunits = a.nblocks * kUnitsPerBlock;
    const int64_t u0 = (int64_t)blockIdx.x * nunits / gridDim.x;
    const int64_t u1 = (int64_t)(blockIdx.x + 1) * nunits / gridDim.x;

    double acc = 0.0;
    int bad = 0;
    // Two register buffers.  Loop invariant at the head: xa holds unit u
    // (loads issued), sa = where unit u lives, sb = where unit u+1 lives.
    float4 xa[kVec], xb[kVec];
    RowSrc sa = {}, sb = {};
    int64_t u = u0;
    if (u < u1) {
        sa = src_of<SRC>(a, u);
        load_unit<SRC>(a, sa, u, tid, xa);
        if (u + 1 < u1) sb = src_of<SRC>(a, u + 1);
    }
    while (u < u1) {
        if (u + 1 < u1) load_unit<SRC>(a, sb, u + 1, tid, xb);
        RowSrc sc = {};
        if (u + 2 < u1) sc = src_of<SRC>(a, u + 2);
        finish_unit<SRC, STORE>(a, sa, u, tid, xa, acc, bad);
        if (++u >= u1) break;
        // xb holds unit u, sb = where it lives, sc = where unit u+1 lives
        if (u + 1 < u1) load_unit<SRC>(a, sc, u + 1, tid, xa);
        RowSrc sd = {};
        if (u + 2 < u1) sd = src_of<SRC>(a, u + 2);
        finish_unit<SRC, STORE>(a, sb, u, tid, xb, acc, bad);
        ++u;
        sa = sc;
        sb = sd;
    }

    // CTA sum in a fixed order
    acc = warp_sum(acc);
    if ((tid & 31) == 0) s_part[tid >> 5] = acc;
    bad = __syncthreads_or(bad);
    if (tid == 0) {
        double t = 0.0;
        for (int w = 0; w < kWarps; ++w) t += s_part[w];
        a.partials[blockIdx.x] = t;
        if (bad) atomicOr(a.found_inf, 1);
        __threadfence();
        const unsigned ticket = atomicAdd(a.counter, 1u);
        s_last = (ticket == gridDim.x - 1);
    }
    __syncthreads();
    if (!s_last) return;

    // the last CTA: add the partials of every CTA in a fixed order
    __threadfence();
    double t = 0.0;
    for (int i = tid; i < (int)gridDim.x; i += kThreads) t += __ldcg(a.partials + i);
    t = warp_sum(t);
    __syncthreads();  // s_part reuse
    if ((tid & 31) == 0) s_part[tid >> 5] = t;
    __syncthreads();
    if (tid == 0) {
        double total = 0.0;
        for (int w = 0; w < kWarps; ++w) total += s_part[w];
        *a.sumsq = *a.sumsq + total;
        *a.counter = 0u;  // ready for the next launch on this workspace
    }
}

// three CTAs of 256 threads per SM, at most one per unit (n blocks: 2n units)
// and one per partial slot
template <typename Layout>
int64_t persistent_grid(const Layout* L, int64_t n)
{
    int64_t grid = (int64_t)L->sm_count * kCtasPerSm;
    if (grid > n * kUnitsPerBlock) grid = n * kUnitsPerBlock;
    if (grid > L->max_partials) grid = L->max_partials;
    return grid;
}

}  // namespace

extern "C" int fp8z1_norm_reset(double* d_sumsq, int32_t* d_found_inf, void* stream)
{
    if (!d_sumsq || !d_found_inf) return FP8Z1_EINVAL;
    if (!fp8z1::aligned(d_sumsq, 8) || !fp8z1::aligned(d_found_inf, 4)) return FP8Z1_EALIGN;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(d_sumsq, 0, sizeof(double), s) != cudaSuccess ||
        cudaMemsetAsync(d_found_inf, 0, sizeof(int32_t), s) != cudaSuccess) {
        cudaGetLastError();
        return FP8Z1_ECUDA;
    }
    return FP8Z1_OK;
}

extern "C" int fp8z1_grad_norm(const fp8z1_layout* L, const float* grad_shard, int64_t b0, int64_t b1,
                               double* d_sumsq, int32_t* d_found_inf, void* stream)
{
    fp8z1::NvtxRange nvtx_range("fp8z1_grad_norm");
    if (!grad_shard || !d_sumsq || !d_found_inf) return FP8Z1_EINVAL;
    const int st = fp8z1::check_range(L, b0, b1);
    if (st != FP8Z1_OK) return st;
    if (!fp8z1::aligned(grad_shard, 16) || !fp8z1::aligned(d_sumsq, 8) || !fp8z1::aligned(d_found_inf, 4))
        return FP8Z1_EALIGN;
    const int64_t n = b1 - b0;
    if (n == 0) return FP8Z1_OK;
    NormArgs a = {};
    a.g = reinterpret_cast<const float4*>(grad_shard);
    a.b0 = b0;
    a.nblocks = n;
    a.partials = L->d_partials;
    a.counter = L->d_counter;
    a.status = L->d_status;
    a.sumsq = d_sumsq;
    a.found_inf = d_found_inf;
    fp8z1::count_launch();
    norm_kernel<kFolded, false><<<(unsigned)persistent_grid(L, n), kThreads, 0,
                                 static_cast<cudaStream_t>(stream)>>>(a);
    return fp8z1::launch_status();
}

extern "C" int fp8z1_fold_norm(const fp8z1_layout* L, const float* const* d_grad_params, float* grad_shard,
                               int64_t b0, int64_t b1, double* d_sumsq, int32_t* d_found_inf, void* stream)
{
    fp8z1::NvtxRange nvtx_range("fp8z1_fold_norm");
    if (!d_grad_params || !d_sumsq || !d_found_inf) return FP8Z1_EINVAL;
    const int st = fp8z1::check_range(L, b0, b1);
    if (st != FP8Z1_OK) return st;
    if (!fp8z1::aligned(d_grad_params, sizeof(void*)) || (grad_shard && !fp8z1::aligned(grad_shard, 16)) ||
        !fp8z1::aligned(d_sumsq, 8) || !fp8z1::aligned(d_found_inf, 4))
        return FP8Z1_EALIGN;
    const int64_t n = b1 - b0;
    if (n == 0) return FP8Z1_OK;
    NormArgs a = {};
    a.lut = L->d_lut;
    a.units = L->d_units;
    a.param_elems = L->d_param_elems;
    a.params = d_grad_params;
    a.store = reinterpret_cast<float4*>(grad_shard);
    a.partials = L->d_partials;
    a.counter = L->d_counter;
    a.status = L->d_status;
    a.sumsq = d_sumsq;
    a.found_inf = d_found_inf;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    auto blocks = [&](int64_t k0, int64_t k1) {  // through the block table
        if (k0 == k1) return;
        a.b0 = k0;
        a.nblocks = k1 - k0;
        const unsigned grid = (unsigned)persistent_grid(L, k1 - k0);
        fp8z1::count_launch();
        if (grad_shard) {
            a.store = reinterpret_cast<float4*>(grad_shard) + (k0 - b0) * (FP8Z1_BLOCK_ELEMS / 4);
            norm_kernel<kRows, true><<<grid, kThreads, 0, s>>>(a);
        } else {
            norm_kernel<kRows, false><<<grid, kThreads, 0, s>>>(a);
        }
    };
    // Without the store, the sum of squares needs no blocks: params the range
    // holds whole are read as flat runs (the layout's run table), and the
    // whole row-block strips of a param it cuts as one contiguous span; only
    // the partial strips at either end go through the block table
    // (fp8z1::norm_pieces).  The pieces are separate launches on one stream,
    // each adding its total to *d_sumsq, in a fixed order: the sum is
    // deterministic for a range.
    if (grad_shard) {
        blocks(b0, b1);
        return fp8z1::launch_status();
    }
    std::vector<fp8z1::NormPiece> pieces;
    try {
        fp8z1::norm_pieces(L, b0, b1, pieces);
    } catch (...) {
        return FP8Z1_ENOMEM;
    }
    for (const fp8z1::NormPiece& pc : pieces) {
        if (pc.kind == fp8z1::NormPiece::kBlocks) {
            blocks(pc.a, pc.b);
        } else if (pc.kind == fp8z1::NormPiece::kWholeParams) {
            const int64_t u0 = L->param_unit0[(size_t)pc.a], u1 = L->param_unit0[(size_t)pc.b];
            a.b0 = u0;
            a.nblocks = u1 - u0;
            fp8z1::count_launch();
            norm_kernel<kParams, false><<<(unsigned)persistent_grid(L, u1 - u0), kThreads, 0, s>>>(a);
        } else {
            a.b0 = 0;
            a.span_param = pc.param;
            a.span_offset = pc.a;
            a.span_elems = pc.b - pc.a;
            a.nblocks = (pc.b - pc.a + FP8Z1_BLOCK_ELEMS - 1) / FP8Z1_BLOCK_ELEMS;
            fp8z1::count_launch();
            norm_kernel<kSpan, false><<<(unsigned)persistent_grid(L, a.nblocks), kThreads, 0, s>>>(a);
        }
    }
    return fp8z1::launch_status();
}

// The grad norm of an MXFP8 shard: a flat range of (g1 - g0) groups of 32
// FP32 grads, in the same reduction.  Its whole 16384-element blocks are read
// as the folded shard is (the fastest of the sources: 0.80 against 0.82 ms for
// the same buffer read as flat runs); a short last block, if any, is a second
// launch that adds its part.
extern "C" int fp8z1_mx_grad_norm(const fp8z1_mx_layout* L, const float* grad_shard, int64_t g0,
                                  int64_t g1, double* d_sumsq, int32_t* d_found_inf, void* stream)
{
    fp8z1::NvtxRange nvtx_range("fp8z1_mx_grad_norm");
    if (!L || !grad_shard || !d_sumsq || !d_found_inf) return FP8Z1_EINVAL;
    if (g0 < 0 || g1 < g0 || g1 > L->n_groups) return FP8Z1_EINVAL;
    if (!L->on_device) return FP8Z1_ENODEV;
    if (!fp8z1::aligned(grad_shard, 16) || !fp8z1::aligned(d_sumsq, 8) || !fp8z1::aligned(d_found_inf, 4))
        return FP8Z1_EALIGN;
    const int64_t n = (g1 - g0) * FP8Z1_MX_GROUP;
    if (n == 0) return FP8Z1_OK;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    NormArgs a = {};
    a.partials = L->d_partials;
    a.counter = L->d_counter;
    a.sumsq = d_sumsq;
    a.found_inf = d_found_inf;
    const int64_t full = n / FP8Z1_BLOCK_ELEMS, rem = n % FP8Z1_BLOCK_ELEMS;
    if (full > 0) {
        a.g = reinterpret_cast<const float4*>(grad_shard);
        a.nblocks = full;
        fp8z1::count_launch();
        norm_kernel<kFolded, false><<<(unsigned)persistent_grid(L, full), kThreads, 0, s>>>(a);
    }
    if (rem > 0) {
        a.g = reinterpret_cast<const float4*>(grad_shard + full * FP8Z1_BLOCK_ELEMS);
        a.span_elems = rem;
        a.nblocks = 1;
        fp8z1::count_launch();
        norm_kernel<kFlat, false><<<(unsigned)persistent_grid(L, 1), kThreads, 0, s>>>(a);
    }
    return fp8z1::launch_status();
}

// ---------------------------------------------------------------------------
// The same reduction for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc at all: a framework whose caching
// allocator already owns the device memory (a foreign cudaMalloc can fail, or
// make the CUDA driver synchronise the device), or a step loop that must never
// block on an allocation.  fp8z1_grad_norm takes its workspace from a layout,
// which fp8z1_build_layout allocates.  This variant takes it from a file-scope
// array instead, so it needs neither a layout nor any allocation.
//
// Workspace: one double per CTA plus the finished-CTA counter, in a static
// array that every device which loads the library holds until the process
// exits (8 * (4096 + 1) bytes).  A call runs the persistent grid of the other
// entry points -- three CTAs per SM, at most one per half block -- so it
// needs one slot per CTA: 4096 slots cover any device with up to 1365 SMs.
// One call covers at most FP8Z1_NOALLOC_MAX_BLOCKS blocks (the header's
// stated bound); larger ranges are rejected -- split them into several
// calls, which accumulate into the same *d_sumsq.
namespace {

constexpr int kNoAllocMaxCtas = 4096;
constexpr int kMaxDevices = 64;

// partials[0, kNoAllocMaxCtas), then the counter (as an unsigned) in the last slot
static __device__ __align__(256) double g_noalloc_scratch[kNoAllocMaxCtas + 1];

// What a device's first call looked up: the workspace's device address, the
// device's SM count, and the CUDA context both belong to (by its unique id).
// A device reset destroys the context and may load the module at another
// address, so a new context id triggers a fresh lookup.
struct NoAllocDevice {
    double* addr = nullptr;
    int sm_count = 0;
    unsigned long long ctx_id = 0;
};

std::mutex g_noalloc_mutex;
NoAllocDevice g_noalloc_dev[kMaxDevices];

// The current context's unique id, through the driver's entry points (the
// library does not link the driver library itself).  0 when it cannot be read.
unsigned long long current_context_id()
{
    using GetCurrent = int (*)(void**);
    using GetId = int (*)(void*, unsigned long long*);
    static GetCurrent get_current = nullptr;
    static GetId get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<GetCurrent>(f);
        f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<GetId>(f);
        cudaGetLastError();
    });
    if (!get_current || !get_id) return 0;
    void* ctx = nullptr;
    unsigned long long id = 0;
    if (get_current(&ctx) != 0 || ctx == nullptr || get_id(ctx, &id) != 0) return 0;
    return id;
}

// The device address of the static workspace on the current device and the
// device's SM count, looked up on the host with that device current (host
// code cannot use the array's name as an address): once per device, and
// again only when the device's context has changed.
int noalloc_workspace(double** out, int* sm_count)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return FP8Z1_ECUDA;
    }
    if (dev < 0 || dev >= kMaxDevices) return FP8Z1_ECUDA;
    // 0 before the device's context exists: the lookup below creates it
    const unsigned long long ctx = current_context_id();
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    NoAllocDevice& d = g_noalloc_dev[dev];
    if (d.addr == nullptr || ctx == 0 || ctx != d.ctx_id) {
        void* p = nullptr;
        int sms = 0;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1) {
            cudaGetLastError();
            d = NoAllocDevice();
            return FP8Z1_ECUDA;
        }
        d.addr = static_cast<double*>(p);
        d.sm_count = sms;
        d.ctx_id = current_context_id();
    }
    *out = d.addr;
    *sm_count = d.sm_count;
    return FP8Z1_OK;
}

}  // namespace

extern "C" int fp8z1_grad_norm_noalloc(const float* grad_shard, int64_t n_blocks, double* d_sumsq,
                                       int32_t* d_found_inf, void* stream)
{
    fp8z1::NvtxRange nvtx_range("fp8z1_grad_norm_noalloc");
    if (!grad_shard || !d_sumsq || !d_found_inf || n_blocks < 0) return FP8Z1_EINVAL;
    if (n_blocks > FP8Z1_NOALLOC_MAX_BLOCKS) return FP8Z1_EINVAL;  // beyond the stated bound
    if (!fp8z1::aligned(grad_shard, 16) || !fp8z1::aligned(d_sumsq, 8) || !fp8z1::aligned(d_found_inf, 4))
        return FP8Z1_EALIGN;
    if (n_blocks == 0) return FP8Z1_OK;
    double* partials = nullptr;
    int sm_count = 0;
    const int st = noalloc_workspace(&partials, &sm_count);
    if (st != FP8Z1_OK) return st;
    unsigned* counter = reinterpret_cast<unsigned*>(partials + kNoAllocMaxCtas);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // the counter must start at zero; the partials are written before they are read
    if (cudaMemsetAsync(counter, 0, sizeof(unsigned), s) != cudaSuccess) {
        cudaGetLastError();
        return FP8Z1_ECUDA;
    }
    NormArgs a = {};
    a.g = reinterpret_cast<const float4*>(grad_shard);
    a.nblocks = n_blocks;
    a.partials = partials;
    a.counter = counter;
    a.sumsq = d_sumsq;
    a.found_inf = d_found_inf;
    int64_t grid = (int64_t)sm_count * kCtasPerSm;
    if (grid > n_blocks * kUnitsPerBlock) grid = n_blocks * kUnitsPerBlock;
    if (grid > kNoAllocMaxCtas) grid = kNoAllocMaxCtas;
    fp8z1::count_launch();
    norm_kernel<kFolded, false><<<(unsigned)grid, kThreads, 0, s>>>(a);
    return fp8z1::launch_status();
}

FP8Z1_CHECKED_MISSES_READER(checked_misses_norm)
