// Bounds checks of a checked build (FP8Z1_CHECKED=1): every load or store a
// kernel makes to a row-major param is tested against the param's extent
// (E * R * C elements, from the layout); an access outside is skipped and
// counted in this translation unit's device counter, which the host reads
// through fp8z1_checked_misses.  In a release build the test is a constant
// true and nothing is counted.
#pragma once

#include "internal.h"

namespace fp8z1 {

#if FP8Z1_CHECKED
// one counter per translation unit (each is its own device module)
static __device__ unsigned long long g_checked_misses;
#endif

// Whether elements [first, first + width) of a param of `elems` elements all
// exist; a miss is counted (checked builds).
__device__ __forceinline__ bool in_extent(int64_t first, int width, int64_t elems)
{
#if FP8Z1_CHECKED
    if (first < 0 || first + width > elems) {
        atomicAdd(&g_checked_misses, 1ull);
        return false;
    }
#else
    (void)first;
    (void)width;
    (void)elems;
#endif
    return true;
}

}  // namespace fp8z1

// The host reader of this translation unit's counter (checked builds).
#if FP8Z1_CHECKED
#define FP8Z1_CHECKED_MISSES_READER(name)                                                \
    uint64_t fp8z1::name()                                                               \
    {                                                                                    \
        unsigned long long v = 0;                                                        \
        if (cudaMemcpyFromSymbol(&v, fp8z1::g_checked_misses, sizeof v) != cudaSuccess) { \
            cudaGetLastError();                                                          \
            return ~0ull;                                                                \
        }                                                                                \
        return v;                                                                        \
    }
#else
#define FP8Z1_CHECKED_MISSES_READER(name)
#endif
