// AllGather-GEMM instantiations of the fused kernel: chunk transfer on the copy engine
// (no in-kernel workers), on TMA bulk copies, or on vector loads/stores; bf16 or fp32 C;
// one CTA or a CTA pair per tile.
#include "dt_internal.h"

namespace dt {

namespace {
template <int COPY, bool F32>
cudaError_t launch_copy(const KParams& p, int grid, bool cooperative, cudaStream_t stream,
                        bool pair) {
  return pair ? launch_fused<kOpAG, COPY, F32, true>(p, grid, cooperative, stream)
              : launch_fused<kOpAG, COPY, F32, false>(p, grid, cooperative, stream);
}
}  // namespace

cudaError_t launch_ag_kernel(const KParams& p, int copy_mode, bool f32, int grid,
                             bool cooperative, cudaStream_t stream, bool pair) {
  switch (copy_mode) {
    case kCopyNone:
      return f32 ? launch_copy<kCopyNone, true>(p, grid, cooperative, stream, pair)
                 : launch_copy<kCopyNone, false>(p, grid, cooperative, stream, pair);
    case kCopyTma:
      return f32 ? launch_copy<kCopyTma, true>(p, grid, cooperative, stream, pair)
                 : launch_copy<kCopyTma, false>(p, grid, cooperative, stream, pair);
    case kCopyLdst:
      return f32 ? launch_copy<kCopyLdst, true>(p, grid, cooperative, stream, pair)
                 : launch_copy<kCopyLdst, false>(p, grid, cooperative, stream, pair);
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace dt
