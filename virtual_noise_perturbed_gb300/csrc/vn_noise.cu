// vn_noise.cu -- the noise dump and the mean-abs reduction metric.
//
// Noise dump: the "_cpu_normal_noise" contract of the EvoX API page
// "evox.triton_kernels.kernels.virtual_noise": out[i, t] = PRNG(seed_i, offset + t).
// Reduction metric: the page's "virtual_reduce_metric":
//   fitness[i] = mean_k |center[k] + sigma * PRNG(seed_i, offset + k)|.
//
// Both are bound by the integer hash (about 20 32-bit integer operations per
// element) and, for the dump, by the 4-byte store per element. Each thread
// works on groups of 4 consecutive elements so that the state of the next
// element is the previous one plus GAMMA (a two-operation 64-bit add) and the
// dump writes one 16-byte store per group.
#include <cooperative_groups.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "vn_hash.cuh"
#include "vn_internal.h"

namespace cg = cooperative_groups;

namespace vn {
namespace {

constexpr int kDumpThreads = 256;
constexpr int kDumpGroups = 8;                                  // groups of 4 per thread
constexpr int64_t kDumpStride = kDumpThreads * 4;               // columns between a thread's groups
constexpr int64_t kDumpChunk = kDumpStride * kDumpGroups;       // elements per CTA step
// GAMMA * kDumpStride mod 2^64: the state difference between a thread's consecutive groups.
constexpr uint64_t kDumpStep = kGamma * static_cast<uint64_t>(kDumpStride);
// GAMMA * (kDumpStride - 3): from a group's last element to the next group's first.
constexpr uint64_t kDumpGroupHop = kGamma * static_cast<uint64_t>(kDumpStride - 3);

// Grid-stride over (row i, chunk of kDumpChunk columns). Thread t makes the
// 4-element groups at columns c + 4t + 1024g, g < 8: one 16-byte store per group,
// consecutive lanes on consecutive 16-byte segments. The state of the next
// element is the previous plus GAMMA; in a chunk that lies inside its row one
// state chain runs through the thread's groups (the step after a group's last
// element adds (1024 - 3)*GAMMA, landing on the next group's first), and at a
// ragged row end the next group's state is the previous group's plus
// 1024*GAMMA, so no 64-bit multiply is needed per group.
// vec4: every row starts 16-byte aligned (out aligned and n % 4 == 0).
// kIdx32: the chunk count fits in 32 bits, so the row of a chunk is a 32-bit
// division (a 64-bit one costs several instructions per element).
// One dump value of the state st: the uniform's exact noise, or the Gaussian variant.
template <int kKind>
__device__ __forceinline__ float dump_value(uint64_t st) {
  if constexpr (kKind == kGaussian) {
    return kGaussScale *
           noise_value<kGaussian>(static_cast<uint32_t>(st), static_cast<uint32_t>(st >> 32));
  } else {
    return noise_from_bits(mix_to_one_plus_u(st));
  }
}

template <bool kIdx32, int kKind>
__global__ void __launch_bounds__(kDumpThreads)
noise_dump_kernel(const int64_t* __restrict__ seeds, int64_t n, uint64_t offset,
                  float* __restrict__ out, int64_t chunks_per_row, int64_t total_chunks,
                  int vec4, uint32_t g_lo, uint32_t g_hi, uint32_t one) {
  // g_lo:g_hi = GAMMA and one = 1, passed at run time: the carry half of the
  // state step is then a multiply-add on the IMAD pipe (add64_madc).
  for (int64_t c = blockIdx.x; c < total_chunks; c += gridDim.x) {
    const int64_t i = kIdx32 ? static_cast<int64_t>(static_cast<uint32_t>(c) /
                                                    static_cast<uint32_t>(chunks_per_row))
                             : c / chunks_per_row;
    const int64_t t0 = (c - i * chunks_per_row) * kDumpChunk + threadIdx.x * 4;
    const uint64_t seed = static_cast<uint64_t>(__ldg(seeds + i));
    float* row = out + i * n;
    uint64_t gst = index_term(offset + static_cast<uint64_t>(t0)) + seed;  // first element of the group
    if (vec4 && t0 - threadIdx.x * 4 + kDumpChunk <= n) {
      // The whole chunk lies inside the row: no per-group checks. One state chain
      // runs through the thread's groups: the step after a group's last element
      // adds (kDumpStride - 3) * GAMMA, which lands on the next group's first.
      uint32_t slo = static_cast<uint32_t>(gst), shi = static_cast<uint32_t>(gst >> 32);
#pragma unroll
      for (int g = 0; g < kDumpGroups; ++g) {
        float v[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          v[q] = dump_value<kKind>((static_cast<uint64_t>(shi) << 32) | slo);
          if (q < 3)
            add64_madc(slo, shi, g_lo, g_hi, one);
          else if (g + 1 < kDumpGroups)
            add64_madc(slo, shi, static_cast<uint32_t>(kDumpGroupHop), static_cast<uint32_t>(kDumpGroupHop >> 32), one);
        }
        __stcs(reinterpret_cast<float4*>(row + t0 + g * kDumpStride),
               make_float4(v[0], v[1], v[2], v[3]));
      }
      continue;
    }
    // number of this thread's groups that start inside the row
    const int64_t left = n - t0;
    const int full = left <= 0 ? 0 : static_cast<int>((left + kDumpStride - 1) / kDumpStride < kDumpGroups ? (left + kDumpStride - 1) / kDumpStride : kDumpGroups);
#pragma unroll
    for (int g = 0; g < kDumpGroups; ++g) {
      if (g < full) {
        const int64_t t = t0 + g * kDumpStride;
        uint64_t st = gst;
        float v[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          v[q] = dump_value<kKind>(st);
          st += kGamma;
        }
        if (vec4 && t + 4 <= n) {
          __stcs(reinterpret_cast<float4*>(row + t), make_float4(v[0], v[1], v[2], v[3]));
        } else {
#pragma unroll
          for (int q = 0; q < 4; ++q)
            if (t + q < n) row[t + q] = v[q];
        }
        gst += kDumpStep;
      }
    }
  }
}

constexpr int kMetricThreads = 256;

// Individual i is handled by the S CTAs of a cluster (S = gridDim.y, 1 when the
// population alone fills the GPU); CTA rank s sums |center[k] + sigma*n| over its
// slice of k, thread t over k = k0 + 4t + 1024g + q. Partial sums are added in a
// fixed order: lanes by shuffle, warps in order, then the S CTAs' sums in rank
// order through distributed shared memory. Grid-stride over individuals.
template <bool kCluster>
__global__ void __launch_bounds__(kMetricThreads)
reduce_metric_kernel(const float* __restrict__ center, const int64_t* __restrict__ seeds,
                     int64_t pop, int64_t n, float sigma, float inv_n, uint64_t offset,
                     float* __restrict__ fitness, int vec4, uint32_t g_lo, uint32_t g_hi,
                     uint32_t one) {
  __shared__ float s_warp[kMetricThreads / 32];
  __shared__ float s_cta;
  const int slices = gridDim.y;
  // slice bounds, multiples of 4 so that 16-byte loads stay aligned
  const int64_t per = ((n + slices - 1) / slices + 3) / 4 * 4;
  const int64_t k_begin = min(n, static_cast<int64_t>(blockIdx.y) * per);
  const int64_t k_end = min(n, k_begin + per);
  for (int64_t i = blockIdx.x; i < pop; i += gridDim.x) {
    const uint64_t seed = static_cast<uint64_t>(__ldg(seeds + i));
    float acc = 0.f;
    for (int64_t k = k_begin + static_cast<int64_t>(threadIdx.x) * 4; k < k_end;
         k += kMetricThreads * 4) {
      uint64_t st = index_term(offset + static_cast<uint64_t>(k)) + seed;
      if (vec4 && k + 4 <= k_end) {  // the common case: four in-range elements, no checks
        const float4 c4 = __ldg(reinterpret_cast<const float4*>(center + k));
        const float c[4] = {c4.x, c4.y, c4.z, c4.w};
        uint32_t slo = static_cast<uint32_t>(st), shi = static_cast<uint32_t>(st >> 32);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          acc += fabsf(fmaf(sigma, noise_from_bits(mix_to_one_plus_u(slo, shi)), c[q]));
          add64_madc(slo, shi, g_lo, g_hi, one);
        }
      } else {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          if (k + q < k_end)
            acc += fabsf(fmaf(sigma, noise_from_bits(mix_to_one_plus_u(st)), __ldg(center + k + q)));
          st += kGamma;
        }
      }
    }
#pragma unroll
    for (int s = 16; s > 0; s >>= 1) acc += __shfl_down_sync(0xffffffffu, acc, s);
    if ((threadIdx.x & 31) == 0) s_warp[threadIdx.x >> 5] = acc;
    __syncthreads();
    if (threadIdx.x == 0) {
      float total = 0.f;
#pragma unroll
      for (int w = 0; w < kMetricThreads / 32; ++w) total += s_warp[w];
      s_cta = total;
    }
    if constexpr (!kCluster) {
      if (threadIdx.x == 0) fitness[i] = s_cta * inv_n;
      __syncthreads();
    } else {
      cg::cluster_group cluster = cg::this_cluster();
      cluster.sync();
      if (cluster.block_rank() == 0 && threadIdx.x == 0) {
        float total = 0.f;
        for (int q = 0; q < slices; ++q) total += *cluster.map_shared_rank(&s_cta, q);
        fitness[i] = total * inv_n;
      }
      cluster.sync();  // no CTA may leave (or reuse s_cta) while rank 0 reads it
    }
  }
}

}  // namespace

template <int kKind>
void dump_launch(bool idx32, unsigned grid, cudaStream_t stream, const int64_t* seeds, int64_t n,
                 uint64_t offset, float* out, int64_t chunks_per_row, int64_t total, int vec4) {
  if (idx32)
    noise_dump_kernel<true, kKind><<<grid, kDumpThreads, 0, stream>>>(
        seeds, n, offset, out, chunks_per_row, total, vec4, kGammaLo, kGammaHi, 1u);
  else
    noise_dump_kernel<false, kKind><<<grid, kDumpThreads, 0, stream>>>(
        seeds, n, offset, out, chunks_per_row, total, vec4, kGammaLo, kGammaHi, 1u);
}

cudaError_t launch_noise_dump(const int64_t* seeds, int64_t pop, int64_t n, uint64_t offset,
                              int kind, float* out, cudaStream_t stream) {
  DeviceInfo dev;
  cudaError_t err = device_info(&dev);
  if (err != cudaSuccess) return err;
  const int64_t chunks_per_row = (n + kDumpChunk - 1) / kDumpChunk;
  const int64_t total = pop * chunks_per_row;
  const int vec4 = (n % 4 == 0) && (reinterpret_cast<uintptr_t>(out) % 16 == 0);
  const int64_t grid = std::min<int64_t>(total, static_cast<int64_t>(dev.sm_count) * 8);
  const bool idx32 = total <= 0xFFFFFFFFll;
  if (kind == kGaussian)
    dump_launch<kGaussian>(idx32, static_cast<unsigned>(grid), stream, seeds, n, offset, out,
                           chunks_per_row, total, vec4);
  else
    dump_launch<kUniform>(idx32, static_cast<unsigned>(grid), stream, seeds, n, offset, out,
                          chunks_per_row, total, vec4);
  return cudaGetLastError();
}

cudaError_t launch_reduce_metric(const float* center, const int64_t* seeds, int64_t pop,
                                 int64_t n, float sigma, float inv_n, uint64_t offset,
                                 float* fitness, cudaStream_t stream) {
  DeviceInfo dev;
  cudaError_t err = device_info(&dev);
  if (err != cudaSuccess) return err;
  const int vec4 = (reinterpret_cast<uintptr_t>(center) % 16 == 0);
  const int64_t resident = static_cast<int64_t>(dev.sm_count) * 8;
  // Split each individual over a cluster while the population alone leaves the
  // GPU mostly idle and each slice keeps at least 16 Ki elements.
  int slices = 1;
  while (slices < 8 && pop * slices < resident && n >= static_cast<int64_t>(slices) * 2 * 16384)
    slices *= 2;
  // With more individuals than resident CTAs, whole individuals per CTA can leave
  // the last round mostly idle (4096 individuals on 1216 CTAs: 4 rounds, the
  // last a third full); halves of individuals balance the rounds better (7
  // rounds, 96 % full: 2.6 % faster there).
  if (slices == 1 && n >= 2 * 2 * 16384) {
    auto fill = [&](int64_t units) {
      const int64_t rounds = (units + resident - 1) / resident;
      return static_cast<double>(units) / static_cast<double>(rounds * resident);
    };
    if (fill(pop) < 0.9 && fill(2 * pop) > fill(pop)) slices = 2;
  }
  if (slices == 1) {
    const int64_t grid = std::min<int64_t>(pop, resident);
    reduce_metric_kernel<false><<<static_cast<unsigned>(grid), kMetricThreads, 0, stream>>>(
        center, seeds, pop, n, sigma, inv_n, offset, fitness, vec4, kGammaLo, kGammaHi, 1u);
    return cudaGetLastError();
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(std::min<int64_t>(pop, std::max<int64_t>(1, resident / slices))),
                     static_cast<unsigned>(slices), 1);
  cfg.blockDim = dim3(kMetricThreads, 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = static_cast<unsigned>(slices);
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, reduce_metric_kernel<true>, center, seeds, pop, n, sigma, inv_n,
                            offset, fitness, vec4, kGammaLo, kGammaHi, 1u);
}

}  // namespace vn
