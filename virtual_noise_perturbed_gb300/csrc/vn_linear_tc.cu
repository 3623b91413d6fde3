// vn_linear_tc.cu -- tcgen05/TMEM perturbed linear (placeholder until the
// tensor-core kernel lands): reports that the path does not apply.
#include <cuda_runtime.h>

#include "vn_internal.h"

namespace vn {

__device__ unsigned int g_device_status = 0;

bool linear_tc_applies(const void*, vn_dtype, const void*, vn_dtype, int64_t, int64_t, int64_t) {
  return false;
}

cudaError_t launch_linear_tc(const LinearArgs&, cudaStream_t) { return cudaErrorNotSupported; }

cudaError_t take_device_status(unsigned int* status, cudaStream_t stream) {
  cudaError_t err = cudaMemcpyFromSymbolAsync(status, g_device_status, sizeof(unsigned int), 0,
                                              cudaMemcpyDeviceToHost, stream);
  if (err != cudaSuccess) return err;
  err = cudaStreamSynchronize(stream);
  if (err != cudaSuccess) return err;
  if (*status != 0) {
    const unsigned int zero = 0;
    err = cudaMemcpyToSymbolAsync(g_device_status, &zero, sizeof(zero), 0,
                                  cudaMemcpyHostToDevice, stream);
    if (err == cudaSuccess) err = cudaStreamSynchronize(stream);
  }
  return err;
}

}  // namespace vn
