// AllGather-GEMM instantiations of the fused kernel: chunk transfer on the copy engine
// (no in-kernel workers), on TMA bulk copies, or on vector loads/stores; bf16 or fp32 C;
// one CTA or a CTA pair per tile.
#include "dt_internal.h"

namespace dt {

namespace {
template <int COPY, bool F32>
cudaError_t launch_copy(const KParams& p, int grid, bool cooperative, cudaStream_t stream, int cl) {
  switch (cl) {
    case 1: return launch_fused<kOpAG, COPY, F32, 1>(p, grid, cooperative, stream);
    case 2: return launch_fused<kOpAG, COPY, F32, 2>(p, grid, cooperative, stream);
    default: return cudaErrorInvalidValue;
  }
}
}  // namespace

cudaError_t launch_ag_kernel(const KParams& p, int copy_mode, bool f32, int grid,
                             bool cooperative, cudaStream_t stream, int cl) {
  switch (copy_mode) {
    case kCopyNone:
      return f32 ? launch_copy<kCopyNone, true>(p, grid, cooperative, stream, cl)
                 : launch_copy<kCopyNone, false>(p, grid, cooperative, stream, cl);
    case kCopyTma:
      return f32 ? launch_copy<kCopyTma, true>(p, grid, cooperative, stream, cl)
                 : launch_copy<kCopyTma, false>(p, grid, cooperative, stream, cl);
    case kCopyLdst:
      return f32 ? launch_copy<kCopyLdst, true>(p, grid, cooperative, stream, cl)
                 : launch_copy<kCopyLdst, false>(p, grid, cooperative, stream, cl);
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace dt
