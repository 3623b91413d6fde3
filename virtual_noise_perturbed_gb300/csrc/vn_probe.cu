// vn_probe.cu -- the hash alone, as a measurement kernel (not a step of the method).
//
//   sums[t] = sum_{e < m} PRNG(seed, offset + t*m + e),  t < n_sums
//
// in fp32 as two partial sums, one over the even e and one over the odd e (each in
// order of e), added at the end.
//
// PRNG is the noise of the EvoX API page "evox.triton_kernels.kernels.virtual_noise"
// (entries "_splitmix64_step", "_cpu_normal_noise"; state reading in vn_hash.cuh).
// Every thread regenerates its m consecutive elements in registers and writes one
// float, so the launch costs the hash and little else. Per element:
//   - the state step: a 64-bit add, one ALU add and one IMAD carry-add;
//   - the finalizer: 12 ALU-pipe and 6 IMAD-pipe operations on 32-bit halves,
//     counting the state add's low word;
//   - half a packed two-lane fp32 add for the -1.5 and half of one for the sum.
// That is the least the other kernels spend besides the hash, so its element rate is
// the measured ceiling of the integer ALU pipe for this hash. The other kernels'
// rooflines are read against it, beside the figure derived from the pipe's width
// and the clock.
#include <cuda_runtime.h>

#include <algorithm>

#include "vn_hash.cuh"
#include "vn_internal.h"

namespace vn {
namespace {

constexpr int kProbeThreads = 256;
constexpr int kProbeUnroll = 8;

__global__ void __launch_bounds__(kProbeThreads)
hash_probe_kernel(uint64_t seed, uint64_t offset, int64_t n_sums, int64_t m,
                  float* __restrict__ sums, uint32_t g_lo, uint32_t g_hi, uint32_t one) {
  const int64_t t = static_cast<int64_t>(blockIdx.x) * kProbeThreads + threadIdx.x;
  if (t >= n_sums) return;
  const uint64_t st = seed + index_term(offset + static_cast<uint64_t>(t) * static_cast<uint64_t>(m));
  uint32_t slo = static_cast<uint32_t>(st), shi = static_cast<uint32_t>(st >> 32);
  float2 acc = make_float2(0.f, 0.f);  // the even and the odd elements' partial sums
  const float2 shift = make_float2(-1.5f, -1.5f);
  int64_t e = 0;
  for (; e + kProbeUnroll <= m; e += kProbeUnroll) {
#pragma unroll
    for (int q = 0; q < kProbeUnroll; q += 2) {
      float2 r;
      r.x = __uint_as_float(mix_to_one_plus_u(slo, shi));
      add64_madc(slo, shi, g_lo, g_hi, one);
      r.y = __uint_as_float(mix_to_one_plus_u(slo, shi));
      add64_madc(slo, shi, g_lo, g_hi, one);
      acc = __fadd2_rn(acc, __fadd2_rn(r, shift));
    }
  }
  for (; e < m; ++e) {
    const float v = noise_from_bits(mix_to_one_plus_u(slo, shi));
    if (e & 1)
      acc.y += v;
    else
      acc.x += v;
    add64_madc(slo, shi, g_lo, g_hi, one);
  }
  sums[t] = acc.x + acc.y;
}

}  // namespace

cudaError_t launch_hash_probe(uint64_t seed, uint64_t offset, int64_t n_sums, int64_t m,
                              float* sums, cudaStream_t stream) {
  const int64_t grid = (n_sums + kProbeThreads - 1) / kProbeThreads;
  hash_probe_kernel<<<static_cast<unsigned>(grid), kProbeThreads, 0, stream>>>(
      seed, offset, n_sums, m, sums, kGammaLo, kGammaHi, 1u);
  return cudaGetLastError();
}

}  // namespace vn
