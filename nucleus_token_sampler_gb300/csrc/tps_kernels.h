// tps_kernels.h -- host addresses of the sampler kernels.  Each (kernel, element type) pair is
// instantiated in a translation unit of its own (tps_k_*.cu) so that the four compile in
// parallel; the launch code in tps_api.cu takes them through these functions.
#pragma once

#include <cstdint>

#include "tps_common.cuh"

namespace tps {

using ClusterKernel = void (*)(Args);
using StreamKernel = void (*)(Args, int, uint32_t);

ClusterKernel cluster_kernel_f32();
ClusterKernel cluster_kernel_bf16();
StreamKernel stream_kernel_f32();
StreamKernel stream_kernel_bf16();

}  // namespace tps
