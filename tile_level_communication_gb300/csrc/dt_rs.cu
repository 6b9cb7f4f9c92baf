// GEMM-ReduceScatter instantiations of the fused kernel (bf16 or fp32 out_s).
#include "dt_internal.h"

namespace dt {

namespace {
template <bool F32>
cudaError_t launch_one(const KParams& p, int grid, cudaStream_t stream) {
  auto kern = fused_gemm_kernel<kOpRS, kCopyNone, F32>;
  const int smem = kernel_smem_bytes(true, kCopyNone);
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
  cfg.attrs = nullptr;
  cfg.numAttrs = 0;
  return cudaLaunchKernelEx(&cfg, kern, p);
}
}  // namespace

cudaError_t launch_rs_kernel(const KParams& p, bool f32, int grid, cudaStream_t stream) {
  return f32 ? launch_one<true>(p, grid, stream) : launch_one<false>(p, grid, stream);
}

}  // namespace dt
