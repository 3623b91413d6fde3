// vn_internal.h -- launchers shared between the C-ABI layer (vn_api.cu) and
// the kernel translation units. Arguments reaching these functions have been
// validated by the C-ABI layer: pointers non-null and aligned, sizes >= 1 and
// their products below 2^63.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "vn.h"
#include "vn_smem.h"

namespace vn {

// Cached per-device facts (SM count, compute capability, opt-in shared memory).
struct DeviceInfo {
  int device = -1;
  int sm_count = 0;
  int cc_major = 0;
  int cc_minor = 0;
  int smem_optin = 0;
};
cudaError_t device_info(DeviceInfo* info);

// out[i, t] = PRNG(seed_i, offset + t), t < n; kind: VN_NOISE_UNIFORM (the
// centered uniform, exact) or VN_NOISE_GAUSSIAN (the Box-Muller variant).
cudaError_t launch_noise_dump(const int64_t* seeds, int64_t pop, int64_t n, uint64_t offset,
                              int kind, float* out, cudaStream_t stream);

// out[e] = scale * sum_i fitness[i] * PRNG(seed_i, offset + e), e < m, with the noise of `kind`;
// with theta != NULL also theta[e] = fma(lr, out[e], theta[e]).
cudaError_t launch_grad(const float* fitness, const int64_t* seeds, int64_t pop, int64_t m,
                        uint64_t offset, float scale, int kind, float* out, cudaStream_t stream,
                        float* theta = nullptr, float lr = 0.f);

// fitness[i] = inv_n * sum_k |center[k] + sigma * PRNG(seed_i, offset + k)|.
cudaError_t launch_reduce_metric(const float* center, const int64_t* seeds, int64_t pop,
                                 int64_t n, float sigma, float inv_n, uint64_t offset,
                                 float* fitness, cudaStream_t stream);

struct LinearArgs {
  const void* x;
  vn_dtype x_dt;
  int x_shared;
  const void* w;
  vn_dtype w_dt;
  const void* b;  // may be null
  vn_dtype b_dt;
  const int64_t* seeds;
  int64_t pop, batch, in, out;
  float sigma;
  uint64_t offset;
  void* y;
  vn_dtype y_dt;
  vn_act act;
  int kind = 0;  // noise kind: 0 the centered uniform, 1 the Gaussian variant
};

// CUDA-core forward: any dtypes, any batch.
cudaError_t launch_linear_ffma(const LinearArgs& a, cudaStream_t stream);

// Whether the tcgen05 forward can run these arguments (shape/alignment/dtype).
bool linear_tc_applies(const void* x, vn_dtype x_dt, const void* w, vn_dtype w_dt,
                       int64_t batch, int64_t in, int64_t out);
// tcgen05/TMEM forward (x bf16).
cudaError_t launch_linear_tc(const LinearArgs& a, cudaStream_t stream);
// The same with every barrier wait bounded by timeout_ns and, when
// withhold_stage >= 0, one hashing thread of CTA 0 skipping its arrive at that
// stage (test hook for the bounded-wait path).
cudaError_t launch_linear_tc_hook(const LinearArgs& a, cudaStream_t stream, long long withhold_stage,
                                  unsigned long long timeout_ns);

// A chain of perturbed linear layers in one launch (fp32 weights, batch <= 8).
constexpr int kMlpMaxLayers = 8;
constexpr int64_t kMlpMaxBatch = 8;
struct MlpArgs {
  const void* x;
  vn_dtype x_dt;
  int x_shared;
  int n_layers;
  const int64_t* dims;       // host, n_layers + 1
  const float* const* w;     // host array of device pointers
  const float* const* b;     // host array of device pointers (entries may be null)
  const uint64_t* offsets;   // host, n_layers
  const int64_t* seeds;
  int64_t pop, batch;
  float sigma;
  vn_act act;        // between layers
  float* y;
  vn_act act_last = VN_ACT_NONE;  // after the last layer (a single perturbed linear's own)
  int kind = 0;                   // noise kind: 0 the centered uniform, 1 the Gaussian variant
};
// Floats per (individual, batch row) of one activation buffer for these dims.
size_t mlp_buffer_floats(int n_layers, const int64_t* dims);
// Shared memory the kernel needs for one individual at this batch (both buffers).
inline size_t mlp_bytes_per_individual(int64_t batch, size_t buf_floats) {
  const int64_t nb = batch <= 1 ? 1 : batch <= 2 ? 2 : batch <= 4 ? 4 : 8;
  return 2 * static_cast<size_t>(nb) * buf_floats * sizeof(float) + 64;
}
cudaError_t launch_mlp(const MlpArgs& m, cudaStream_t stream);

// out[i] = rank of fitness[i] (ascending, ties by index) / (pop - 1) - 0.5.
cudaError_t launch_centered_ranks(const float* fitness, int64_t pop, float* out,
                                  cudaStream_t stream);
// theta[k] += lr * grad[k], k < n.
cudaError_t launch_es_update(float* theta, const float* grad, int64_t n, float lr,
                             cudaStream_t stream);

// sums[t] = sum_{e < m} PRNG(seed, offset + t*m + e), t < n_sums: the hash alone.
cudaError_t launch_hash_probe(uint64_t seed, uint64_t offset, int64_t n_sums, int64_t m,
                              float* sums, cudaStream_t stream);

// Reads and clears the device status word of the bounded-wait kernels (0 = fine).
cudaError_t take_device_status(unsigned int* status, cudaStream_t stream);

}  // namespace vn
