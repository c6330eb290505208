// Launch-cost diagnostic: an empty kernel launched as the decode kernels are.
// Semantics of the entry point are in include/paged_kv.h.
#include <cuda_runtime.h>

#include "paged_kv.h"
#include "status.h"

namespace {

constexpr int kMaxDevices = 64;
constexpr int kMaxSmemPerCta = 227 * 1024;  // dynamic shared memory a CTA may opt into on sm_103a

__global__ void trace_empty_kernel() {}

bool g_configured[kMaxDevices] = {};

cudaError_t launch_empty(int ctas, int threads, int smem_bytes, cudaStream_t stream) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  if (!g_configured[dev]) {
    err = cudaFuncSetAttribute(trace_empty_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxSmemPerCta);
    if (err != cudaSuccess) return err;
    g_configured[dev] = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(ctas));
  cfg.blockDim = dim3(unsigned(threads));
  cfg.dynamicSmemBytes = size_t(smem_bytes);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, trace_empty_kernel);
}

}  // namespace

extern "C" pkv_status_t pkv_trace_empty_grid(int ctas, int threads, int smem_bytes, void* stream) {
  if (ctas < 1 || threads < 1 || threads > 1024 || smem_bytes < 0 || smem_bytes > kMaxSmemPerCta)
    return pkv::fail(PKV_ERR_INVALID_ARG, "trace_empty_grid: ctas >= 1, threads 1..1024, smem 0..227 KB");
  const cudaError_t err = launch_empty(ctas, threads, smem_bytes, static_cast<cudaStream_t>(stream));
  if (err != cudaSuccess) return pkv::fail(PKV_ERR_CUDA, "trace_empty_grid launch: %s", cudaGetErrorString(err));
  return pkv::ok();
}
