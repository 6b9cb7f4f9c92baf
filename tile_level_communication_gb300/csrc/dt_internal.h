// Declarations shared by the library's translation units (not part of the C ABI).
#pragma once

#include <cuda_runtime.h>

#include <cstdlib>

#include "dt.h"
#include "dt_kernel.cuh"

namespace dt {

// Fused AllGather-GEMM on a caller-supplied scratch buffer using only the in-kernel chunk
// transfer (TMA bulk or ld/st; AUTO means TMA).  Creates no stream, event or host-side
// record: every call clears the scratch's error word and layout tag, so the prepare kernel
// rebuilds the tile order and zeroes the flags and counters, and the call runs with epoch 1.
// Defined in dt_capi.cu; used by the fixed-scratch entry point in dt_static_ws.cu.
dt_status ag_gemm_on_scratch(const void* const* a_shards, const void* b, void* c, void* scratch,
                             size_t scratch_bytes, const dt_args* a, cudaStream_t stream);

// Set the calling thread's dt_last_error() message.
void set_last_error(const char* msg);

// Launch the fused persistent kernel; defined in dt_ag.cu (AllGather variants), dt_rs.cu
// (ReduceScatter / AllReduce variants) and dt_a2a.cu (AllToAll variants).  `cooperative`
// guarantees that every CTA is resident, which the in-kernel chunk transfer relies on.
// `cl`: CTAs per cluster, 1 or 2 (a CTA pair per 256-row tile); grid and copy_ctas are
// multiples of it and the grid is capped at the clusters the GPU holds at once.
cudaError_t launch_ag_kernel(const KParams& p, int copy_mode, bool f32, int grid,
                             bool cooperative, cudaStream_t stream, int cl);
cudaError_t launch_rs_kernel(const KParams& p, bool f32, int grid, cudaStream_t stream, int cl);
cudaError_t launch_a2a_kernel(const KParams& p, bool f32, int grid, cudaStream_t stream, int cl);

// One launch of an instance of the fused kernel (dynamic shared memory raised once).
// Per device and kernel instance: the dynamic shared memory limit raised, and how many of its
// clusters the device holds at once (0 until known).
constexpr int kMaxDevices = 64;
template <int OP, int COPY, bool F32, int CL>
struct LaunchState {
  bool configured[kMaxDevices];
  int max_clusters[kMaxDevices];
};

// Whether the fused kernel is launched with programmatic stream serialization, so that its
// launch and set-up overlap the prepare kernel before it in the stream (the kernel waits for
// that grid before it touches global memory): on unless DT_PDL=0.
inline bool pdl_setting() {
  static const bool v = [] {
    const char* e = getenv("DT_PDL");
    return e ? atoi(e) != 0 : true;
  }();
  return v;
}

template <int OP, int COPY, bool F32, int CL>
cudaError_t launch_fused(const KParams& p, int grid, bool cooperative, cudaStream_t stream) {
  auto kern = fused_gemm_kernel<OP, COPY, F32, CL>;
  const int smem = kernel_smem_bytes(CL);
  static LaunchState<OP, COPY, F32, CL> state = {};
  int dev = 0;
  cudaError_t de = cudaGetDevice(&dev);
  if (de != cudaSuccess) return de;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  if (!state.configured[dev]) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    state.configured[dev] = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  if (CL > 1) {
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CL;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    // a persistent cluster launch is sized to the clusters the GPU holds at once, so every CTA
    // is resident (what the in-kernel chunk transfer needs; checked here rather than with the
    // cooperative attribute, which a profiler cannot replay together with clusters); the
    // tiles are spread over whatever grid runs
    int& max_clusters = state.max_clusters[dev];
    if (max_clusters < 1) {
      cudaLaunchConfig_t probe = cfg;
      probe.gridDim = dim3(CL);
      cudaError_t e = cudaOccupancyMaxActiveClusters(&max_clusters, kern, &probe);
      if (e != cudaSuccess) return e;
      if (max_clusters < 1) return cudaErrorInvalidConfiguration;
    }
    if (grid > CL * max_clusters) cfg.gridDim = dim3(CL * max_clusters);
    if (cooperative && p.copy_ctas >= static_cast<int>(cfg.gridDim.x))
      return cudaErrorCooperativeLaunchTooLarge;
  } else if (cooperative) {
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  // not with the cooperative attribute, and not while a debug timeline is attached (its reset
  // is a memset between the prepare kernel and this one)
  if (pdl_setting() && !(CL == 1 && cooperative) && p.trace == nullptr) {
    attr[cfg.numAttrs].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[cfg.numAttrs].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs += 1;
  }
  return cudaLaunchKernelEx(&cfg, kern, p);
}

}  // namespace dt
