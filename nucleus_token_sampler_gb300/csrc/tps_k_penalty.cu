// The penalty kernel on float32 and bfloat16 logits, and its launch (its own translation unit).
#include "tps_penalty.cuh"

namespace tps {

cudaError_t launch_penalties(const PenaltyArgs& a, bool bf16, int sms, cudaStream_t stream)
{
    auto k = bf16 ? &penalty_rows_kernel<__nv_bfloat16> : &penalty_rows_kernel<float>;
    const size_t smem = 2 * (size_t)penalty_slots(a.H) * sizeof(uint32_t);
    if (smem > 48 * 1024) {  // long histories: opt in to the larger table (on the current device)
        const cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    // One CTA per row, up to 64 per SM (grid-stride beyond): the block scheduler hands rows to SMs
    // as earlier ones finish (four 512-thread CTAs fit an SM when their tables do).
    const int64_t cap = (int64_t)sms * 64;
    const int64_t grid = a.B < cap ? a.B : cap;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3(kPenaltyThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    return cudaLaunchKernelEx(&cfg, k, a);
}

}  // namespace tps
