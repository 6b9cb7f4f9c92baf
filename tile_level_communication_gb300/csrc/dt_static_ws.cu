// Fused AllGather-GEMM for callers that cannot allocate device memory.
//
// Some callers have no way to provide the workspace that dt_ag_gemm needs: a plugin whose
// host framework owns all device memory and hands it no scratch, a serving process that
// reserved the whole GPU for its own allocator, or a latency-critical path that cannot afford
// the device-wide synchronisation of cudaMalloc.  dt_ag_gemm_static_scratch serves them: its
// scratch (tile order, ready flags, piece counters, gather buffer) is a fixed device array
// defined in this file, so the call allocates nothing.
//
// Cost and limits: every GPU that loads this part of the library holds DT_STATIC_SCRATCH_BYTES
// until the process exits; problems whose workspace (dt_workspace_size) exceeds it are
// rejected.  Every call on a device shares the one array and leaves its contents behind, so
// calls that overlap on the GPU (two streams, or two host threads) race and must be ordered
// by the caller.
#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>

#include "dt.h"
#include "dt_internal.h"

// The scratch itself.  In host code this name is a host-side stand-in, never a device
// address: host code must obtain the address with cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_static_scratch[DT_STATIC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_setup_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Once per device, with that device current: resolve the scratch's device address.
dt_status scratch_address(int dev, void** out) {
  if (dev < 0 || dev >= kMaxDevices) {
    dt::set_last_error("fixed scratch: device ordinal beyond the supported 64");
    return DT_ERR_UNSUPPORTED;
  }
  std::lock_guard<std::mutex> lk(g_setup_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* ptr = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&ptr, g_static_scratch);
    if (e != cudaSuccess || ptr == nullptr) {
      dt::set_last_error("fixed scratch: cudaGetSymbolAddress failed");
      return DT_ERR_CUDA;
    }
    g_scratch_addr[dev] = ptr;
  }
  *out = g_scratch_addr[dev];
  return DT_OK;
}

}  // namespace

extern "C" dt_status dt_ag_gemm_static_scratch(const void* const* a_shards, const void* b,
                                               void* c, const dt_args* a, void* stream) {
  if (!a) return DT_ERR_INVALID;
  const size_t need = dt_workspace_size(a, DT_OP_AG_GEMM);
  if (need == 0) return DT_ERR_INVALID;  // dt_last_error() names the bad argument
  if (need > DT_STATIC_SCRATCH_BYTES) {
    dt::set_last_error("fixed scratch: this problem needs more workspace than the "
                       "DT_STATIC_SCRATCH_BYTES (32 MiB) array holds; use dt_ag_gemm");
    return DT_ERR_WORKSPACE;
  }
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return DT_ERR_CUDA;
  void* scratch = nullptr;
  const dt_status s = scratch_address(dev, &scratch);
  if (s != DT_OK) return s;
  return dt::ag_gemm_on_scratch(a_shards, b, c, scratch, DT_STATIC_SCRATCH_BYTES, a,
                                reinterpret_cast<cudaStream_t>(stream));
}

// The array starts with the same error block as a workspace, so dt_check reads and clears it.
extern "C" dt_status dt_static_scratch_check(void* stream, uint32_t* info) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return DT_ERR_CUDA;
  void* scratch = nullptr;
  const dt_status s = scratch_address(dev, &scratch);
  if (s != DT_OK) return s;
  return dt_check(scratch, stream, info);
}
