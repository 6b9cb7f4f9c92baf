// GEMM-ReduceScatter / GEMM-AllReduce instantiations of the fused kernel (bf16 or fp32
// out, one CTA or a CTA pair per tile).
#include "dt_internal.h"

namespace dt {

cudaError_t launch_rs_kernel(const KParams& p, bool f32, int grid, cudaStream_t stream, bool pair) {
  if (pair)
    return f32 ? launch_fused<kOpRS, kCopyNone, true, true>(p, grid, false, stream)
               : launch_fused<kOpRS, kCopyNone, false, true>(p, grid, false, stream);
  return f32 ? launch_fused<kOpRS, kCopyNone, true, false>(p, grid, false, stream)
             : launch_fused<kOpRS, kCopyNone, false, false>(p, grid, false, stream);
}

}  // namespace dt
