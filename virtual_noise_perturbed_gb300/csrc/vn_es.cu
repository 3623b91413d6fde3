// vn_es.cu -- the two ES steps around the gradient estimate that are not noise
// work: fitness shaping by centered ranks, and the parameter update.
//
// Centered ranks ("fitness = centered ranks in [-0.5, 0.5]", the shaping of the
// ES policy and gradient-only workloads): out[i] = rank_i / (pop - 1) - 0.5 with
// rank_i the position of fitness[i] in ascending order, equal values ordered by
// index. The order is a total order on float bit patterns (negative values
// below positive ones, -0 below +0, NaNs at the ends by sign), so every input
// gives a permutation of 0..pop-1. rank_i is counted exactly as an integer and
// converted to fp32 by round-to-nearest-even (exact up to 2^24 individuals, rounded
// above); the conversion, the division and the subtraction are single fp32
// operations, so the result is fully determined.
//
// Update: theta[k] += lr * grad[k] (one fp32 fma per element), the ascent step
// on the estimate of the page's module description.
//
// Ranking is a count per element over the whole population (pop^2
// comparisons): the keys are staged in shared memory 2048 at a time and the
// threads sharing an i split them. At the workloads' populations (1,024 and
// 16,384) that is 1e6 and 2.7e8 comparisons.
#include <cuda_runtime.h>

#include <algorithm>

#include "vn_internal.h"

namespace vn {
namespace {

constexpr int kRankThreads = 256;
constexpr int kRankTile = 2048;

// Float bits -> an unsigned key whose order is the float order (total).
__device__ __forceinline__ uint32_t order_key(float f) {
  const uint32_t b = __float_as_uint(f);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// kTpi threads share one i: each scans every kTpi-th key of a staged tile and
// the kTpi partial counts are added with shuffles, so a population of a
// thousand still spreads over a hundred CTAs.
template <int kTpi>
__global__ void __launch_bounds__(kRankThreads)
centered_ranks_kernel(const float* __restrict__ fitness, int pop, float* __restrict__ out) {
  __shared__ uint32_t s_key[kRankTile];
  constexpr int kPerCta = kRankThreads / kTpi;
  const int sub = threadIdx.x % kTpi;
  // 64-bit: the last CTA's first index may pass 2^31 - 1 when pop is close to it.
  const int64_t i = static_cast<int64_t>(blockIdx.x) * kPerCta + threadIdx.x / kTpi;
  const uint32_t ki = i < pop ? order_key(fitness[i]) : 0u;
  uint32_t rank = 0;
  for (int j0 = 0; j0 < pop; j0 += kRankTile) {
    const int jn = min(kRankTile, pop - j0);
    __syncthreads();
    for (int t = threadIdx.x; t < jn; t += kRankThreads) s_key[t] = order_key(fitness[j0 + t]);
    __syncthreads();
    // Keys below ki, and equal keys at a lower index (j < i <=> t < i - j0).
    const int64_t before = i - j0;
#pragma unroll 8
    for (int t = sub; t < jn; t += kTpi) {
      const uint32_t kj = s_key[t];
      rank += (kj < ki) | ((kj == ki) & (t < before));
    }
  }
#pragma unroll
  for (int o = kTpi / 2; o > 0; o >>= 1) rank += __shfl_xor_sync(0xffffffffu, rank, o);
  if (i < pop && sub == 0) {
    const float denom = static_cast<float>(pop > 1 ? pop - 1 : 1);
    out[i] = static_cast<float>(rank) / denom - 0.5f;
  }
}

__global__ void es_update_kernel(float* __restrict__ theta, const float* __restrict__ grad,
                                 int64_t n, float lr, int vec4) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (vec4) {
    const int64_t n4 = n / 4;
    for (int64_t v = t; v < n4; v += stride) {
      float4 p = reinterpret_cast<float4*>(theta)[v];
      const float4 g = __ldg(reinterpret_cast<const float4*>(grad) + v);
      p.x = fmaf(lr, g.x, p.x);
      p.y = fmaf(lr, g.y, p.y);
      p.z = fmaf(lr, g.z, p.z);
      p.w = fmaf(lr, g.w, p.w);
      reinterpret_cast<float4*>(theta)[v] = p;
    }
    for (int64_t e = n4 * 4 + t; e < n; e += stride) theta[e] = fmaf(lr, grad[e], theta[e]);
  } else {
    for (int64_t e = t; e < n; e += stride) theta[e] = fmaf(lr, grad[e], theta[e]);
  }
}

}  // namespace

template <int kTpi>
cudaError_t launch_ranks(const float* fitness, int64_t pop, float* out, cudaStream_t stream) {
  constexpr int kPerCta = kRankThreads / kTpi;
  const int64_t grid = (pop + kPerCta - 1) / kPerCta;
  centered_ranks_kernel<kTpi><<<static_cast<unsigned>(grid), kRankThreads, 0, stream>>>(
      fitness, static_cast<int>(pop), out);
  return cudaGetLastError();
}

// Threads per i: the most that still leaves every thread at least 64 keys to scan,
// except a full warp per i from 1,024 individuals on (32 keys or more per thread; at
// 1,024 individuals it cuts the launch from 8.1 to 6.2 µs).
cudaError_t launch_centered_ranks(const float* fitness, int64_t pop, float* out,
                                  cudaStream_t stream) {
  if (pop >= 32 * 32) return launch_ranks<32>(fitness, pop, out, stream);
  if (pop >= 8 * 64) return launch_ranks<8>(fitness, pop, out, stream);
  if (pop >= 2 * 64) return launch_ranks<2>(fitness, pop, out, stream);
  return launch_ranks<1>(fitness, pop, out, stream);
}

cudaError_t launch_es_update(float* theta, const float* grad, int64_t n, float lr,
                             cudaStream_t stream) {
  DeviceInfo dev;
  cudaError_t err = device_info(&dev);
  if (err != cudaSuccess) return err;
  const int vec4 = (reinterpret_cast<uintptr_t>(theta) % 16 == 0) &&
                   (reinterpret_cast<uintptr_t>(grad) % 16 == 0);
  const int64_t per = vec4 ? (n + 3) / 4 : n;
  const int64_t grid = std::max<int64_t>(
      1, std::min<int64_t>((per + 255) / 256, static_cast<int64_t>(dev.sm_count) * 8));
  es_update_kernel<<<static_cast<unsigned>(grid), 256, 0, stream>>>(theta, grad, n, lr, vec4);
  return cudaGetLastError();
}

}  // namespace vn
