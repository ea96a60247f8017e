// Entry points of the fused optimizer step (fp8z1_step, fp8z1_step_fused,
// fp8z1_step_fused_dev): argument checks, the per-step scalars, and the
// launches of the step kernels of step_kernel.cuh.
//
// "面向 Blockwise FP8 量化的 ZeRO 优化器设计" §总结: the optimizer update is
// elementwise on the rank's slice, then each rank quantises new FP8 params
// and their scales; "DeepSpeed ZeRO 优化" §三 / §六 / §七: unscale and clip,
// then the update; a found inf skips the step.
#include <algorithm>
#include <vector>

#include "step_args.h"

namespace {

using namespace fp8z1;
using namespace fp8z1::stepk;

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

// The launches of a step over [b0, b1): runs of blocks of params made of full
// tiles only (precomputed with the layout) go to the kernel without the
// padding test, everything else to the one with it.
void launch_segments(const fp8z1_layout* L, StepArgs a, int64_t b0, int64_t b1, cudaStream_t s,
                     unsigned forms)
{
    auto one = [&](int64_t k0, int64_t k1, bool pad) {
        a.blk_off = k0 - b0;
        fp8z1::count_launch();
        if (pad)
            launch<true>(a, k1 - k0, s, forms);
        else
            launch<false>(a, k1 - k0, s, forms);
    };
    int64_t k = b0;
    for (size_t r = 0; r + 1 < L->full_runs.size() && k < b1; r += 2) {
        const int64_t lo = std::max(L->full_runs[r], k), hi = std::min(L->full_runs[r + 1], b1);
        if (lo >= hi) continue;
        if (lo > k) one(k, lo, true);
        one(lo, hi, false);
        k = hi;
    }
    if (k < b1) one(k, b1, true);
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
#if FP8Z1_CHECKED
    a.param_elems = L->d_param_elems;
#endif
    a.b0 = b0;
    a.status = L->d_status;
    a.c = scalars(hp);
    launch_segments(L, a, b0, b1, static_cast<cudaStream_t>(stream), kCodesFolded);
    return fp8z1::launch_status();
}

namespace {

int step_fused_impl(const fp8z1_layout* L, const fp8z1_adamw_hp* hp, const fp8z1_adamw_hp* hp_if_set,
                    const int32_t* d_select, const StepScalars* h_scalars, StepScalars* d_scalars,
                    const float* grad_shard, const float* const* d_grad_params, float* master_shard,
                    float* m_shard, float* v_shard, uint8_t* fp8_shard, uint8_t* const* d_fp8_params,
                    float* scale_shard, float* block_cos, uint32_t* block_underflow, int64_t b0, int64_t b1,
                    const double* d_sumsq, const int32_t* d_found_inf, void* stream)
{
    // exactly one scalar source: hp by value (optionally a second set picked
    // by *d_select), or d_scalars
    if ((hp == nullptr) == (d_scalars == nullptr)) return FP8Z1_EINVAL;
    if ((hp_if_set == nullptr) != (d_select == nullptr)) return FP8Z1_EINVAL;
    if (hp_if_set && (block_cos || !in_domain(hp_if_set))) return FP8Z1_EINVAL;
    if (d_select && !fp8z1::aligned(d_select, 4)) return FP8Z1_EALIGN;
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
#if FP8Z1_CHECKED
    a.param_elems = L->d_param_elems;
#endif
    a.b0 = b0;
    a.grad_params = d_grad_params;
    a.code_params = d_fp8_params;
    a.block_cos = block_cos;
    a.block_underflow = block_underflow;
    a.status = L->d_status;
    a.dsc = d_scalars;
    a.select = d_select;
    if (hp) a.c = scalars(hp);
    if (hp_if_set) a.c2 = scalars(hp_if_set);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (h_scalars && cudaMemcpyAsync(d_scalars, h_scalars, sizeof(StepScalars),
                                     cudaMemcpyHostToDevice, s) != cudaSuccess) {
        cudaGetLastError();
        return FP8Z1_ECUDA;
    }
    const unsigned forms = (d_grad_params ? kGradRows : 0u) | (d_fp8_params ? kCodesRows : 0u) |
                           (fp8_shard ? kCodesFolded : 0u) | (block_cos ? kMonitors : 0u) |
                           (d_scalars ? kDevScalars : 0u) | (d_select ? kSelScalars : 0u);
    launch_segments(L, a, b0, b1, s, forms);
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
    return step_fused_impl(L, hp, nullptr, nullptr, nullptr, nullptr, grad_shard, d_grad_params, master_shard,
                           m_shard, v_shard, fp8_shard, d_fp8_params, scale_shard, block_cos, block_underflow, b0,
                           b1, d_sumsq, d_found_inf, stream);
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
    return step_fused_impl(L, nullptr, nullptr, nullptr, h_scalars, d_scalars, grad_shard, d_grad_params,
                           master_shard, m_shard,
                           v_shard, fp8_shard, d_fp8_params, scale_shard, block_cos, block_underflow, b0, b1,
                           d_sumsq, d_found_inf, stream);
}

extern "C" int fp8z1_step_fused_select(const fp8z1_layout* L, const fp8z1_adamw_hp* hp_if_clear,
                                       const fp8z1_adamw_hp* hp_if_set, const int32_t* d_select,
                                       const float* grad_shard, const float* const* d_grad_params,
                                       float* master_shard, float* m_shard, float* v_shard, uint8_t* fp8_shard,
                                       uint8_t* const* d_fp8_params, float* scale_shard, int64_t b0, int64_t b1,
                                       const double* d_sumsq, const int32_t* d_found_inf, void* stream)
{
    fp8z1::NvtxRange nvtx_range("fp8z1_step_fused_select");
    if (!hp_if_clear || !hp_if_set || !d_select) return FP8Z1_EINVAL;
    return step_fused_impl(L, hp_if_clear, hp_if_set, d_select, nullptr, nullptr, grad_shard, d_grad_params,
                           master_shard, m_shard, v_shard, fp8_shard, d_fp8_params, scale_shard, nullptr, nullptr,
                           b0, b1, d_sumsq, d_found_inf, stream);
}

extern "C" int fp8z1_graph_step_nodes(void* graph, void** nodes, int32_t capacity, int32_t* n_nodes)
{
    if (!graph || !n_nodes || capacity < 0 || (capacity > 0 && !nodes)) return FP8Z1_EINVAL;
    cudaGraph_t g = static_cast<cudaGraph_t>(graph);
    size_t n = 0;
    if (cudaGraphGetNodes(g, nullptr, &n) != cudaSuccess) {
        cudaGetLastError();
        return FP8Z1_ECUDA;
    }
    std::vector<cudaGraphNode_t> all(n);
    if (n && cudaGraphGetNodes(g, all.data(), &n) != cudaSuccess) {
        cudaGetLastError();
        return FP8Z1_ECUDA;
    }
    int32_t found = 0;
    for (cudaGraphNode_t node : all) {
        cudaGraphNodeType type;
        if (cudaGraphNodeGetType(node, &type) != cudaSuccess || type != cudaGraphNodeTypeKernel) continue;
        cudaKernelNodeParams kp = {};
        if (cudaGraphKernelNodeGetParams(node, &kp) != cudaSuccess) {
            cudaGetLastError();
            continue;
        }
        if (!is_value_kernel<false>(kp.func) && !is_value_kernel<true>(kp.func)) continue;
        if (found < capacity) nodes[found] = node;
        ++found;
    }
    *n_nodes = found;
    return found > capacity ? FP8Z1_EINVAL : FP8Z1_OK;
}

extern "C" int fp8z1_graph_set_step_hp(void* graph_exec, void* const* nodes, int32_t n_nodes,
                                       const fp8z1_adamw_hp* hp)
{
    if (!graph_exec || n_nodes < 0 || (n_nodes > 0 && !nodes) || !hp || !in_domain(hp)) return FP8Z1_EINVAL;
    cudaGraphExec_t exec = static_cast<cudaGraphExec_t>(graph_exec);
    const StepScalars c = scalars(hp);
    for (int32_t i = 0; i < n_nodes; ++i) {
        cudaGraphNode_t node = static_cast<cudaGraphNode_t>(nodes[i]);
        cudaKernelNodeParams kp = {};
        if (cudaGraphKernelNodeGetParams(node, &kp) != cudaSuccess || !kp.kernelParams ||
            (!is_value_kernel<false>(kp.func) && !is_value_kernel<true>(kp.func))) {
            cudaGetLastError();
            return FP8Z1_EINVAL;
        }
        StepArgs a = *static_cast<const StepArgs*>(kp.kernelParams[0]);
        a.c = c;
        void* args[] = {&a};
        kp.kernelParams = args;
        kp.extra = nullptr;
        if (cudaGraphExecKernelNodeSetParams(exec, node, &kp) != cudaSuccess) {
            cudaGetLastError();
            return FP8Z1_ECUDA;
        }
    }
    return FP8Z1_OK;
}

extern "C" int fp8z1_step_scalars_from_hp(const fp8z1_adamw_hp* hp, fp8z1_step_scalars* out)
{
    if (!hp || !out || !in_domain(hp)) return FP8Z1_EINVAL;
    *out = scalars(hp);
    return FP8Z1_OK;
}
