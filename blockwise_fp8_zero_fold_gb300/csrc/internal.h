// Internal definitions shared by the translation units of libfp8z1.so.
#pragma once

#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>
#include <stdint.h>

#include <atomic>
#include <vector>

#include "fp8z1.h"

// Device-side status bits, OR-ed into the layout's status word by a kernel
// that meets device data it cannot use (it then skips that work).
#define FP8Z1_DEV_BADPTR 1u  // a param pointer was null or not elem_size aligned

// Checked builds (libfp8z1_checked.so, compiled with -DFP8Z1_CHECKED=1) test
// every access a kernel makes to a row-major param against that param's
// extent, skip an access that falls outside and count it (checked.cuh).
#ifndef FP8Z1_CHECKED
#define FP8Z1_CHECKED 0
#endif

// A run of at most FP8Z1_BLOCK_ELEMS consecutive row-major elements of one
// param: what the norm reads for a param that a block range holds whole.
struct fp8z1_unit {
    int64_t offset;  // first element, from the param's start
    int32_t param;
    int32_t count;   // elements, 1 .. FP8Z1_BLOCK_ELEMS
};

struct fp8z1_layout {
    std::vector<fp8z1_shape> shapes;
    std::vector<fp8z1_block> lut;  // host copy of the block lookup table
    int32_t n_params = 0;
    int32_t dp_size = 1;
    int64_t n_blocks = 0;
    int64_t n_real = 0;
    bool on_device = false;
    int device = -1;
    int sm_count = 0;
    fp8z1_block* d_lut = nullptr;      // device copy of `lut`
    double* d_partials = nullptr;      // grad-norm workspace: one double per CTA
    unsigned* d_counter = nullptr;     // grad-norm workspace: CTAs finished
    unsigned* d_status = nullptr;      // FP8Z1_DEV_* bits
    int max_partials = 0;
    std::vector<int64_t> param_block0;  // first block of each param; n_params + 1 entries
    std::vector<int64_t> param_unit0;   // first unit of each param; n_params + 1 entries
    std::vector<fp8z1_unit> units;      // every param cut into units, in param order
    fp8z1_unit* d_units = nullptr;      // device copy of `units`
    int64_t* d_param_elems = nullptr;   // E * R * C of each param (what checked builds test against)
    // [first, last) block pairs, ascending: runs of at least kFullRunMin blocks
    // whose params have R and C multiples of 128 (every block a full tile)
    std::vector<int64_t> full_runs;
    static constexpr int64_t kFullRunMin = 512;
};

// MXFP8 layout: the params' row-major elements back to back, cut into groups
// of 32 consecutive elements (every C a multiple of 32).
struct fp8z1_mx_layout {
    std::vector<fp8z1_shape> shapes;
    int32_t n_params = 0;
    int32_t dp_size = 1;
    int64_t n_groups = 0;
    bool on_device = false;
    int sm_count = 0;
    double* d_partials = nullptr;  // grad-norm workspace: one double per CTA
    unsigned* d_counter = nullptr;
    int max_partials = 0;
};

namespace fp8z1 {

// NVTX ranges around the device entry points, in their own "fp8z1" domain
// (a no-op unless a profiler attaches; ranges of other domains are unaffected).
inline nvtxDomainHandle_t nvtx_domain()
{
    static nvtxDomainHandle_t d = nvtxDomainCreateA("fp8z1");
    return d;
}

struct NvtxRange {
    explicit NvtxRange(const char* name)
    {
        nvtxEventAttributes_t e = {};
        e.version = NVTX_VERSION;
        e.size = NVTX_EVENT_ATTRIB_STRUCT_SIZE;
        e.messageType = NVTX_MESSAGE_TYPE_ASCII;
        e.message.ascii = name;
        nvtxDomainRangePushEx(nvtx_domain(), &e);
    }
    ~NvtxRange() { nvtxDomainRangePop(nvtx_domain()); }
    NvtxRange(const NvtxRange&) = delete;
    NvtxRange& operator=(const NvtxRange&) = delete;
};

// The pieces a grad norm without store reads for blocks [b0, b1), in order:
// block ranges through the block table (partial row-block strips of a cut
// param), runs of params the range holds whole, and contiguous element spans
// of the whole strips of a cut param.  Together they cover every real grad
// element of the range exactly once.
struct NormPiece {
    enum Kind { kBlocks, kWholeParams, kSpan } kind;
    int64_t a, b;   // blocks [a, b) | params [a, b) | elements [a, b) of `param`
    int32_t param;  // kSpan
};
void norm_pieces(const fp8z1_layout* L, int64_t b0, int64_t b1, std::vector<NormPiece>& out);

#if FP8Z1_CHECKED
// Out-of-extent accesses each checked translation unit has counted (and
// skipped) on the current device, since the library was loaded.
uint64_t checked_misses_fold();
uint64_t checked_misses_norm();
uint64_t checked_misses_step_full();
uint64_t checked_misses_step_pad();
#endif

// Kernels this library has enqueued in this process (every device and stream),
// read through fp8z1_kernel_launches.
std::atomic<uint64_t>& launch_counter();
inline void count_launch() { launch_counter().fetch_add(1, std::memory_order_relaxed); }

inline bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Common checks of a layout and a block range for the device entry points.
inline int check_range(const fp8z1_layout* L, int64_t b0, int64_t b1)
{
    if (!L) return FP8Z1_EINVAL;
    if (b0 < 0 || b1 < b0 || b1 > L->n_blocks) return FP8Z1_EINVAL;
    if (!L->on_device) return FP8Z1_ENODEV;
    return FP8Z1_OK;
}

inline int launch_status()
{
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? FP8Z1_OK : FP8Z1_ECUDA;
}

}  // namespace fp8z1
