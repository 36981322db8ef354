// The cluster kernel on bfloat16 logits (its own translation unit; see tps_kernels.h).
#include "tps_cluster.cuh"
#include "tps_kernels.h"

namespace tps {
ClusterKernel cluster_kernel_bf16() { return &sample_rows_kernel<__nv_bfloat16>; }
}  // namespace tps
