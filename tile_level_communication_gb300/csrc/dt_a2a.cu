// GEMM-AllToAll instantiations of the fused kernel (bf16 or fp32 out_h, one CTA or a CTA pair
// per tile), also used by the baseline's per-step launches.
#include "dt_internal.h"

namespace dt {

namespace {
template <bool F32>
cudaError_t launch_cl(const KParams& p, int grid, cudaStream_t stream, int cl) {
  switch (cl) {
    case 1: return launch_fused<kOpA2A, kCopyNone, F32, 1>(p, grid, false, stream);
    case 2: return launch_fused<kOpA2A, kCopyNone, F32, 2>(p, grid, false, stream);
    default: return cudaErrorInvalidValue;
  }
}
}  // namespace

cudaError_t launch_a2a_kernel(const KParams& p, bool f32, int grid, cudaStream_t stream, int cl) {
  return f32 ? launch_cl<true>(p, grid, stream, cl) : launch_cl<false>(p, grid, stream, cl);
}

}  // namespace dt
