// The arguments of the step kernels and their launch, shared by the entry
// points (step.cu) and the two translation units that instantiate the kernels
// (step_full.cu: blocks that are full 128x128 tiles; step_pad.cu: any block,
// skipping the chunks that hold padding only).
#pragma once

#include "update.cuh"

namespace fp8z1 {
namespace stepk {

constexpr int kThreads = 512;
constexpr int kVec = FP8Z1_BLOCK_ELEMS / 4 / kThreads;  // 8 float4 per thread
constexpr int kWarps = kThreads / 32;

// where the grads come from and the codes go (compile-time forms of the kernel)
enum : unsigned {
    kGradRows = 1u,     // grads read row-major through the block table
    kCodesRows = 2u,    // codes written row-major through the block table
    kCodesFolded = 4u,  // codes written to the folded code shard
    kMonitors = 8u,     // per-block underflow count and cosine
    kDevScalars = 16u,  // step scalars read from device memory
    kSelScalars = 32u,  // two scalar sets by value, picked by a device flag
};

// where the kernel takes its step scalars from
enum ScalarSource : int { kScValue = 0, kScDevice = 1, kScSelect = 2 };

struct StepArgs {
    const float4* grad;          // folded grad shard (!kGradRows)
    float4* master;
    float4* mom1;
    float4* mom2;
    uint32_t* codes;             // folded code shard (kCodesFolded)
    float* scales;
    const double* sumsq;
    const int32_t* found_inf;
    const fp8z1_block* lut;
    int64_t b0;                  // the shard's first block: buffers start there
    int64_t blk_off;             // this launch's first block, relative to b0
    const float* const* grad_params;  // kGradRows: row-major FP32 grads
    uint8_t* const* code_params;      // kCodesRows: row-major FP8 params
    unsigned* status;
    float* block_cos;            // kMonitors: cosine(master, dequantised) per block
    uint32_t* block_underflow;   // kMonitors: non-zero masters whose code is 0, per block
    const StepScalars* dsc;      // kDevScalars: the scalars in device memory
    const int32_t* select;       // kSelScalars: c when *select == 0, else c2
    StepScalars c;               // the scalars by value
    StepScalars c2;              // kSelScalars: the other set
#if FP8Z1_CHECKED
    const int64_t* param_elems;  // each param's extent, which row-major accesses are tested against
#endif
};

// One launch of nb blocks from a.blk_off on; `forms` is an OR of the bits above.
template <bool PAD>
void launch(const StepArgs& a, int64_t nb, cudaStream_t s, unsigned forms);

extern template void launch<false>(const StepArgs&, int64_t, cudaStream_t, unsigned);
extern template void launch<true>(const StepArgs&, int64_t, cudaStream_t, unsigned);

// Whether `func` is one of the step kernels taking its scalars by value (the
// ones whose captured graph nodes fp8z1_graph_set_step_hp may rewrite).
template <bool PAD>
bool is_value_kernel(const void* func);

extern template bool is_value_kernel<false>(const void*);
extern template bool is_value_kernel<true>(const void*);

}  // namespace stepk
}  // namespace fp8z1
