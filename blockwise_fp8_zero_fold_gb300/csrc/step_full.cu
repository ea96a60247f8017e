// The step kernels for blocks that are full 128x128 tiles (no padding test).
#include "step_kernel.cuh"

template void fp8z1::stepk::launch<false>(const fp8z1::stepk::StepArgs&, int64_t, cudaStream_t, unsigned);
template bool fp8z1::stepk::is_value_kernel<false>(const void*);

FP8Z1_CHECKED_MISSES_READER(checked_misses_step_full)
