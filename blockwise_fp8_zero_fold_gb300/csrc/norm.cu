// Global grad norm: the sum of squares of the loss-scaled FP32 grads of a
// block range, plus the inf/nan flag.
//
// "DeepSpeed ZeRO 优化" §七 梯度裁剪: the global norm is the square root of the
// sum over every rank of its partial sum of squares (an all-reduce); the clip
// coefficient is formed from it.  §六 / §九 Q6: an inf or nan among the grads
// skips the step.
//
// Accuracy: each square is split exactly into float hi + lo parts
// (x*x and fma(x, x, -x*x)), and a thread adds its 32 squares of a block with
// error-free two-sums, so its per-block partial is within about 32^2 ulp^2 of
// the exact value; partials are then summed in double.  The result is well
// inside 1e-12 relative of the exact sum -- close enough that the clip
// coefficient formed from it rounds to the same FP32 number as one formed from
// the exact sum, except in rare ties.  A thread whose 32 values hold one with
// |x| outside [2^-60, 2^60) (or an inf/nan) redoes them in double, where the
// squares of any finite float are exact.
//
// Reduction: a fixed number of CTAs each take a contiguous run of blocks;
// each writes one double to a workspace, and the last CTA to finish (an atomic
// ticket, no waiting) adds the partials in a fixed order.  The result is
// deterministic for a given device and range.
#include <cuda_runtime.h>

#include <mutex>

#include "internal.h"

namespace {

constexpr int kThreads = 512;
constexpr int kVecPerThread = FP8Z1_BLOCK_ELEMS / 4 / kThreads;  // 8 float4
constexpr int kWarps = kThreads / 32;

__device__ __forceinline__ void two_sum(float a, float b, float& s, float& err)
{
    s = __fadd_rn(a, b);
    const float bb = __fsub_rn(s, a);
    const float aa = __fsub_rn(s, bb);
    err = __fadd_rn(__fsub_rn(a, aa), __fsub_rn(b, bb));
}

// true when x is an inf/nan or too small/large for the float fast path
__device__ __forceinline__ bool out_of_fast_range(float x)
{
    const unsigned u = __float_as_uint(x) & 0x7fffffffu;
    constexpr unsigned kLo = 0x21800000u;  // 2^-60
    constexpr unsigned kHi = 0x5d800000u;  // 2^60
    return u != 0u && (u - kLo) >= (kHi - kLo);
}

__device__ __forceinline__ void add_square(float x, float& hi, float& lo, bool& slow)
{
    slow |= out_of_fast_range(x);
    const float sq = __fmul_rn(x, x);
    const float e = __fmaf_rn(x, x, -sq);  // x*x = sq + e exactly (in range)
    float t;
    two_sum(hi, sq, hi, t);
    lo = __fadd_rn(lo, __fadd_rn(t, e));
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

__global__ void __launch_bounds__(kThreads, 2) grad_norm_kernel(const float4* __restrict__ g,
                                                             int64_t nblocks,
                                                             double* __restrict__ partials,
                                                             unsigned* __restrict__ counter,
                                                             double* __restrict__ d_sumsq,
                                                             int32_t* __restrict__ d_found_inf)
{
    __shared__ double s_part[kWarps];
    __shared__ int s_last;
    const int tid = threadIdx.x;
    const int64_t k0 = (int64_t)blockIdx.x * nblocks / gridDim.x;
    const int64_t k1 = (int64_t)(blockIdx.x + 1) * nblocks / gridDim.x;

    double acc = 0.0;
    int bad = 0;
    for (int64_t k = k0; k < k1; ++k) {
        const float4* p = g + k * (FP8Z1_BLOCK_ELEMS / 4) + tid;
        float4 x[kVecPerThread];
#pragma unroll
        for (int j = 0; j < kVecPerThread; ++j) x[j] = __ldcs(p + j * kThreads);
        float hi = 0.0f, lo = 0.0f;
        bool slow = false;
#pragma unroll
        for (int j = 0; j < kVecPerThread; ++j) {
            add_square(x[j].x, hi, lo, slow);
            add_square(x[j].y, hi, lo, slow);
            add_square(x[j].z, hi, lo, slow);
            add_square(x[j].w, hi, lo, slow);
        }
        if (!slow) {
            acc += (double)hi;
            acc += (double)lo;
        } else {
#pragma unroll
            for (int j = 0; j < kVecPerThread; ++j) {
                add_square_exact(x[j].x, acc, bad);
                add_square_exact(x[j].y, acc, bad);
                add_square_exact(x[j].z, acc, bad);
                add_square_exact(x[j].w, acc, bad);
            }
        }
    }

    // CTA sum in a fixed order
    acc = warp_sum(acc);
    if ((tid & 31) == 0) s_part[tid >> 5] = acc;
    bad = __syncthreads_or(bad);
    if (tid == 0) {
        double t = 0.0;
        for (int w = 0; w < kWarps; ++w) t += s_part[w];
        partials[blockIdx.x] = t;
        if (bad) atomicOr(d_found_inf, 1);
        __threadfence();
        const unsigned ticket = atomicAdd(counter, 1u);
        s_last = (ticket == gridDim.x - 1);
    }
    __syncthreads();
    if (!s_last) return;

    // the last CTA: add the partials of every CTA in a fixed order
    __threadfence();
    double t = 0.0;
    for (int i = tid; i < (int)gridDim.x; i += kThreads) t += __ldcg(partials + i);
    t = warp_sum(t);
    __syncthreads();  // s_part reuse
    if ((tid & 31) == 0) s_part[tid >> 5] = t;
    __syncthreads();
    if (tid == 0) {
        double total = 0.0;
        for (int w = 0; w < kWarps; ++w) total += s_part[w];
        *d_sumsq = *d_sumsq + total;
        *counter = 0u;  // ready for the next launch on this layout
    }
}

}  // namespace

extern "C" int fp8z1_grad_norm(const fp8z1_layout* L, const float* grad_shard, int64_t b0, int64_t b1,
                               double* d_sumsq, int32_t* d_found_inf, void* stream)
{
    if (!grad_shard || !d_sumsq || !d_found_inf) return FP8Z1_EINVAL;
    const int st = fp8z1::check_range(L, b0, b1);
    if (st != FP8Z1_OK) return st;
    if (!fp8z1::aligned(grad_shard, 16) || !fp8z1::aligned(d_sumsq, 8) || !fp8z1::aligned(d_found_inf, 4))
        return FP8Z1_EALIGN;
    const int64_t n = b1 - b0;
    if (n == 0) return FP8Z1_OK;
    // two CTAs of 512 threads per SM, at most one per block and one per partial slot
    int64_t grid = (int64_t)L->sm_count * 2;
    if (grid > n) grid = n;
    if (grid > L->max_partials) grid = L->max_partials;
    grad_norm_kernel<<<(unsigned)grid, kThreads, 0, static_cast<cudaStream_t>(stream)>>>(
        reinterpret_cast<const float4*>(grad_shard), n, L->d_partials, L->d_counter, d_sumsq, d_found_inf);
    return fp8z1::launch_status();
}

// ---------------------------------------------------------------------------
// The same reduction for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc at all: a framework whose caching
// allocator already owns the device memory (a foreign cudaMalloc can fail, or
// make the driver synchronise the device), or a step loop that must never
// block on an allocation.  fp8z1_grad_norm takes its workspace from a layout,
// which fp8z1_build_layout allocates.  This variant takes it from a file-scope
// array instead, so it needs neither a layout nor any allocation.
//
// Workspace: one double per CTA plus the finished-CTA counter, in a static
// array that every device which loads the library holds until the process
// exits (8 * (4096 + 1) bytes).  Each CTA covers up to 64 blocks, so one call
// covers at most 4096 * 64 = 262144 blocks; larger ranges are rejected (split
// them into several calls, which accumulate into the same *d_sumsq).
namespace {

constexpr int64_t kNoAllocBlocksPerCta = 64;
constexpr int kNoAllocMaxCtas = (int)(FP8Z1_NOALLOC_MAX_BLOCKS / kNoAllocBlocksPerCta);
constexpr int kMaxDevices = 64;

// partials[0, kNoAllocMaxCtas), then the counter (as an unsigned) in the last slot
static __device__ __align__(256) double g_noalloc_scratch[kNoAllocMaxCtas + 1];

std::mutex g_noalloc_mutex;
double* g_noalloc_addr[kMaxDevices] = {};

// The device address of the static workspace on the current device, looked up
// once per device (host code cannot use the array's name as an address).
int noalloc_workspace(double** out)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return FP8Z1_ECUDA;
    }
    if (dev < 0 || dev >= kMaxDevices) return FP8Z1_ECUDA;
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    if (g_noalloc_addr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
            cudaGetLastError();
            return FP8Z1_ECUDA;
        }
        g_noalloc_addr[dev] = static_cast<double*>(p);
    }
    *out = g_noalloc_addr[dev];
    return FP8Z1_OK;
}

}  // namespace

extern "C" int fp8z1_grad_norm_noalloc(const float* grad_shard, int64_t n_blocks, double* d_sumsq,
                                       int32_t* d_found_inf, void* stream)
{
    if (!grad_shard || !d_sumsq || !d_found_inf || n_blocks < 0) return FP8Z1_EINVAL;
    if (n_blocks > FP8Z1_NOALLOC_MAX_BLOCKS) return FP8Z1_EINVAL;  // beyond the static workspace
    if (!fp8z1::aligned(grad_shard, 16) || !fp8z1::aligned(d_sumsq, 8) || !fp8z1::aligned(d_found_inf, 4))
        return FP8Z1_EALIGN;
    if (n_blocks == 0) return FP8Z1_OK;
    double* partials = nullptr;
    const int st = noalloc_workspace(&partials);
    if (st != FP8Z1_OK) return st;
    unsigned* counter = reinterpret_cast<unsigned*>(partials + kNoAllocMaxCtas);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // the counter must start at zero; the partials are written before they are read
    if (cudaMemsetAsync(counter, 0, sizeof(unsigned), s) != cudaSuccess) {
        cudaGetLastError();
        return FP8Z1_ECUDA;
    }
    const int64_t grid = (n_blocks + kNoAllocBlocksPerCta - 1) / kNoAllocBlocksPerCta;
    grad_norm_kernel<<<(unsigned)grid, kThreads, 0, s>>>(reinterpret_cast<const float4*>(grad_shard),
                                                         n_blocks, partials, counter, d_sumsq, d_found_inf);
    return fp8z1::launch_status();
}
