// AllGather-GEMM instantiations of the fused kernel: chunk transfer on the copy engine
// (no in-kernel workers), on TMA bulk copies, or on vector loads/stores; bf16 or fp32 C.
#include "dt_internal.h"

namespace dt {

namespace {
template <int COPY, bool F32>
cudaError_t launch_one(const KParams& p, int grid, bool cooperative, cudaStream_t stream) {
  auto kern = fused_gemm_kernel<kOpAG, COPY, F32>;
  const int smem = kernel_smem_bytes(false, COPY);
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = cooperative ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, p);
}
}  // namespace

cudaError_t launch_ag_kernel(const KParams& p, int copy_mode, bool f32, int grid,
                             bool cooperative, cudaStream_t stream) {
  switch (copy_mode) {
    case kCopyNone:
      return f32 ? launch_one<kCopyNone, true>(p, grid, cooperative, stream)
                 : launch_one<kCopyNone, false>(p, grid, cooperative, stream);
    case kCopyTma:
      return f32 ? launch_one<kCopyTma, true>(p, grid, cooperative, stream)
                 : launch_one<kCopyTma, false>(p, grid, cooperative, stream);
    case kCopyLdst:
      return f32 ? launch_one<kCopyLdst, true>(p, grid, cooperative, stream)
                 : launch_one<kCopyLdst, false>(p, grid, cooperative, stream);
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace dt
