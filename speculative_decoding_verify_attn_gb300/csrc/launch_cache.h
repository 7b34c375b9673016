// Host-side launch settings that are per CUDA context and never change once made: the dynamic
// shared-memory limit of a kernel, and the cluster occupancy of a launch shape.  Each is applied or
// queried once per (context, kernel, shape) and remembered, so that a call's host path does not
// repeat a driver round trip that would only return the same answer.  The cache holds no result of
// any computation; a context it has not seen (another device, a caller's own driver-API context,
// a new primary context after a device reset) simply gets the settings made again.
#pragma once

#include <cuda_runtime.h>

namespace specv {

// cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes), once per context
// for each kernel (again only if a later call needs a larger limit).
cudaError_t ensure_dynamic_smem(const void* func, int bytes);

// cudaOccupancyMaxActiveClusters(active, func, cfg), remembered per (context, kernel, cluster size,
// block size, dynamic shared memory).
cudaError_t max_active_clusters(int* active, const void* func, const cudaLaunchConfig_t* cfg);

}  // namespace specv
