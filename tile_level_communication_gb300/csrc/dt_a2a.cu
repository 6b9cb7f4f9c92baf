// GEMM-AllToAll instantiations of the fused kernel (bf16 or fp32 out_h, one CTA or a CTA
// pair per tile), also used by the baseline's per-step launches.
#include "dt_internal.h"

namespace dt {

cudaError_t launch_a2a_kernel(const KParams& p, bool f32, int grid, cudaStream_t stream,
                              bool pair) {
  if (pair)
    return f32 ? launch_fused<kOpA2A, kCopyNone, true, true>(p, grid, false, stream)
               : launch_fused<kOpA2A, kCopyNone, false, true>(p, grid, false, stream);
  return f32 ? launch_fused<kOpA2A, kCopyNone, true, false>(p, grid, false, stream)
             : launch_fused<kOpA2A, kCopyNone, false, false>(p, grid, false, stream);
}

}  // namespace dt
