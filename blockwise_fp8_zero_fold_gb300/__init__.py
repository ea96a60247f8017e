"""blockwise_fp8_zero_fold_gb300: the ZeRO-1 optimizer step for blockwise-FP8
weights (fold/unfold, block LUT, global grad norm, fused unscale + clip +
AdamW + per-block E4M3 quantise) as a C-ABI CUDA library for sm_103a.

``fp8z1`` is the ctypes binding of ``libfp8z1.so``; ``synth`` draws the
seeded synthetic workloads.
"""
