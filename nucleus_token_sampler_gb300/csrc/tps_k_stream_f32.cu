// The streaming kernel on float32 logits (its own translation unit; see tps_kernels.h).
#include "tps_stream.cuh"
#include "tps_kernels.h"

namespace tps {
StreamKernel stream_kernel_f32() { return &stream_rows_kernel<float>; }
}  // namespace tps
