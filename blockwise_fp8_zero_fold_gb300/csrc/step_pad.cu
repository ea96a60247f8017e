// The step kernels for any block, skipping the float4 chunks that hold padding only.
#include "step_kernel.cuh"

template void fp8z1::stepk::launch<true>(const fp8z1::stepk::StepArgs&, int64_t, cudaStream_t, unsigned);
template bool fp8z1::stepk::is_value_kernel<true>(const void*);

FP8Z1_CHECKED_MISSES_READER(checked_misses_step_pad)
