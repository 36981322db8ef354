// The cluster kernel on float32 logits (its own translation unit; see tps_kernels.h).
#include "tps_cluster.cuh"
#include "tps_kernels.h"

namespace tps {
ClusterKernel cluster_kernel_f32() { return &sample_rows_kernel<float>; }
}  // namespace tps
