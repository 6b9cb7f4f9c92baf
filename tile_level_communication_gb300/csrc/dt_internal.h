// Declarations shared by the library's translation units (not part of the C ABI).
#pragma once

#include <cuda_runtime.h>

#include "dt_kernel.cuh"

namespace dt {

// Launch the fused persistent kernel; defined in dt_ag.cu (AllGather variants) and
// dt_rs.cu (ReduceScatter variants).  `cooperative` guarantees that every CTA is resident,
// which the in-kernel chunk transfer relies on.
cudaError_t launch_ag_kernel(const KParams& p, int copy_mode, bool f32, int grid,
                             bool cooperative, cudaStream_t stream);
cudaError_t launch_rs_kernel(const KParams& p, bool f32, int grid, cudaStream_t stream);

}  // namespace dt
