// The rejection-draw kernel on float32 and bfloat16 logits, and its launch (its own translation unit).
#include "tps_reject.cuh"

namespace tps {

cudaError_t launch_reject(const RejectArgs& ra, bool bf16, int sms, cudaStream_t stream)
{
    auto k = bf16 ? &reject_rows_kernel<__nv_bfloat16> : &reject_rows_kernel<float>;
    // One CTA per row (several per SM), grid-stride beyond.
    const int64_t cap = (int64_t)sms * 4;
    const int64_t grid = ra.a.B < cap ? ra.a.B : cap;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = sizeof(Shared);
    cfg.stream = stream;
    return cudaLaunchKernelEx(&cfg, k, ra);
}

}  // namespace tps
