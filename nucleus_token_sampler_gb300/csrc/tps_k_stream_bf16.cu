// The streaming kernel on bfloat16 logits (its own translation unit; see tps_kernels.h).
#include "tps_stream.cuh"
#include "tps_kernels.h"

namespace tps {
StreamKernel stream_kernel_bf16() { return &stream_rows_kernel<__nv_bfloat16>; }
}  // namespace tps
