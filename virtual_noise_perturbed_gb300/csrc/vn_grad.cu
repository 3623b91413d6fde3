// vn_grad.cu -- the ES gradient estimate, bound by regenerating the noise.
//
// EvoX API page "evox.triton_kernels.kernels.virtual_noise", entries
// "virtual_weight_gradient" and "virtual_bias_gradient":
//   grad[e] = sum_i fitness_i * PRNG(seed_i, offset + e) / (pop * sigma)
// with e = j*in + k for a weight block and e = j for a bias block (whose
// offset already points at the bias region). Both are the same flat reduction
// over the population, so one kernel serves both.
//
// Work decomposition
//   * A CTA owns a tile of 256 consecutive elements; lane l of every warp owns
//     elements [8l, 8l + 8) of the tile. The per-element part of the state,
//     (offset + e + 1) * GAMMA, is computed once; per individual the state is
//     that plus the seed (one 64-bit add), then the finalizer; each pair of
//     elements then takes one packed two-lane add (the noise's -1.5) and one
//     packed two-lane FMA into its two sums (each lane rounding as fadd / fmaf).
//   * The 8 warps of the CTA split the CTA's share of the population
//     (individuals are staged in shared memory 256 at a time and read back as
//     one 16-byte broadcast per individual), and their partial sums are added
//     in warp order through shared memory.
//   * When the element count is too small to fill the GPU, the population is
//     further split across the S CTAs of a thread-block cluster (S <= 8); the
//     S partial tiles are added through distributed shared memory in rank
//     order. Every sum is taken in a fixed order, so the result is
//     deterministic for a given device and shape.
//   * With a parameter vector theta (the fused ES step), the thread that
//     stores grad[e] also applies theta[e] = fma(lr, grad[e], theta[e]): the
//     same values as a separate update launch, without it.
#include <cooperative_groups.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>

#include "vn_hash.cuh"
#include "vn_internal.h"

namespace cg = cooperative_groups;

namespace vn {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kE = 8;           // consecutive elements per lane
constexpr int kTile = 32 * kE;  // elements per CTA tile
constexpr int kStage = 256;     // individuals staged per round

template <bool kCluster, int kKind, bool kUpdate>
__global__ void __launch_bounds__(kThreads)
grad_kernel(const float* __restrict__ fitness, const int64_t* __restrict__ seeds, int64_t pop,
            int64_t m, uint64_t offset, float scale, float* __restrict__ out, int64_t tiles,
            float* __restrict__ theta, float lr) {
  __shared__ uint4 s_ind[kStage];  // {seed lo, seed hi, fitness bits, 0}
  __shared__ float s_part[kWarps][kTile];
  __shared__ float s_red[kTile];

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int slices = gridDim.y;
  const int64_t per = (pop + slices - 1) / slices;
  const int64_t p0 = (static_cast<int64_t>(blockIdx.y) * per < pop ? static_cast<int64_t>(blockIdx.y) * per : pop);
  const int64_t p1 = (p0 + per < pop ? p0 + per : pop);

  for (int64_t tile = blockIdx.x; tile < tiles; tile += gridDim.x) {
    const int64_t e0 = tile * kTile + lane * kE;
    uint32_t blo[kE], bhi[kE];  // (offset + e + 1) * GAMMA for this lane's elements
    index_term(offset + static_cast<uint64_t>(e0), blo[0], bhi[0]);
#pragma unroll
    for (int e = 1; e < kE; ++e) {
      blo[e] = blo[e - 1];
      bhi[e] = bhi[e - 1];
      add64(blo[e], bhi[e], kGammaLo, kGammaHi);
    }
    float acc[kE];
#pragma unroll
    for (int e = 0; e < kE; ++e) acc[e] = 0.f;

    for (int64_t c0 = p0; c0 < p1; c0 += kStage) {
      const int cn = static_cast<int>(p1 - c0 < kStage ? p1 - c0 : kStage);
      __syncthreads();
      if (threadIdx.x < cn) {
        const uint64_t s = static_cast<uint64_t>(seeds[c0 + threadIdx.x]);
        s_ind[threadIdx.x] = make_uint4(static_cast<uint32_t>(s), static_cast<uint32_t>(s >> 32),
                                        __float_as_uint(fitness[c0 + threadIdx.x]), 0u);
      }
      __syncthreads();
      for (int q = warp; q < cn; q += kWarps) {
        const uint4 v = s_ind[q];
        // (the Gaussian variant's constant factor rides on the fitness weight)
        const float f = kKind == kGaussian ? kGaussScale * __uint_as_float(v.z) : __uint_as_float(v.z);
        // Element pairs: the noise values' -1.5 and the weighted sum each as one packed
        // two-lane operation (each lane rounds as fadd / fmaf do).
        const float2 f2 = make_float2(f, f);
#pragma unroll
        for (int e = 0; e < kE; e += 2) {
          float2 nz;
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            uint32_t lo = blo[e + h], hi = bhi[e + h];
            add64(lo, hi, v.x, v.y);
            float r;
            if constexpr (kKind == kGaussian)
              r = noise_value<kGaussian>(lo, hi);
            else
              r = __uint_as_float(mix_to_one_plus_u(lo, hi));
            if (h == 0) nz.x = r; else nz.y = r;
          }
          if constexpr (kKind != kGaussian) nz = __fadd2_rn(nz, make_float2(-1.5f, -1.5f));
          const float2 s = __ffma2_rn(f2, nz, make_float2(acc[e], acc[e + 1]));
          acc[e] = s.x;
          acc[e + 1] = s.y;
        }
      }
    }

    // Warp partials -> one partial per element, added in warp order.
#pragma unroll
    for (int e = 0; e < kE; ++e) s_part[warp][lane * kE + e] = acc[e];
    __syncthreads();
    float part = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) part += s_part[w][threadIdx.x];
    __syncthreads();  // s_part is rewritten by the next tile

    if constexpr (!kCluster) {
      const int64_t e = tile * kTile + threadIdx.x;
      if (e < m) {
        const float g = part * scale;
        out[e] = g;
        if constexpr (kUpdate) theta[e] = fmaf(lr, g, theta[e]);
      }
    } else {
      cg::cluster_group cluster = cg::this_cluster();
      s_red[threadIdx.x] = part;
      cluster.sync();
      // Rank r finishes elements [r*kTile/S, (r+1)*kTile/S) of the tile.
      const int rank = static_cast<int>(cluster.block_rank());
      const int span = kTile / slices;
      if (threadIdx.x < span) {
        const int t = rank * span + threadIdx.x;
        float sum = 0.f;
        for (int q = 0; q < slices; ++q) sum += cluster.map_shared_rank(s_red, q)[t];
        const int64_t e = tile * kTile + t;
        if (e < m) {
          const float g = sum * scale;
          out[e] = g;
          if constexpr (kUpdate) theta[e] = fmaf(lr, g, theta[e]);
        }
      }
      cluster.sync();  // no CTA may leave (or reuse s_red) while others read it
    }
  }
}

// Resident CTAs of `fn` per SM on device `dev`, queried once per (kernel,
// device) and kept in `cache` (0 = not yet queried): devices of different
// models in one process get their own figure.
int occupancy(const void* fn, int dev, std::atomic<int> (&cache)[kMaxDevices]) {
  const int known = cache[dev].load(std::memory_order_relaxed);
  if (known > 0) return known;
  int blocks = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, fn, kThreads, 0) != cudaSuccess ||
      blocks < 1)
    blocks = 1;
  cache[dev].store(blocks, std::memory_order_relaxed);
  return blocks;
}

template <int kKind, bool kUpdate>
cudaError_t launch_grad_kind(const float* fitness, const int64_t* seeds, int64_t pop, int64_t m,
                             uint64_t offset, float scale, float* out, float* theta, float lr,
                             cudaStream_t stream) {
  DeviceInfo dev;
  cudaError_t err = device_info(&dev);
  if (err != cudaSuccess) return err;
  const int64_t tiles = (m + kTile - 1) / kTile;
  static std::atomic<int> occ_cache[kMaxDevices];
  const int occ = occupancy(reinterpret_cast<const void*>(&grad_kernel<false, kKind, kUpdate>),
                            dev.device, occ_cache);
  const int64_t resident = static_cast<int64_t>(dev.sm_count) * occ;

  // Split the population across a cluster while the tiles alone leave the GPU
  // mostly idle and each slice keeps at least 64 individuals per warp round.
  int slices = 1;
  while (slices < 8 && tiles * slices < resident &&
         pop >= static_cast<int64_t>(slices) * 2 * 64)
    slices *= 2;

  if (slices == 1) {
    const int64_t grid = std::min<int64_t>(tiles, resident * 4);
    grad_kernel<false, kKind, kUpdate><<<static_cast<unsigned>(grid), kThreads, 0, stream>>>(
        fitness, seeds, pop, m, offset, scale, out, tiles, theta, lr);
    return cudaGetLastError();
  }
  const int64_t grid_x = std::min<int64_t>(tiles, std::max<int64_t>(1, resident * 4 / slices));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid_x), static_cast<unsigned>(slices), 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = static_cast<unsigned>(slices);
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, grad_kernel<true, kKind, kUpdate>, fitness, seeds, pop, m,
                            offset, scale, out, tiles, theta, lr);
}

}  // namespace

cudaError_t launch_grad(const float* fitness, const int64_t* seeds, int64_t pop, int64_t m,
                        uint64_t offset, float scale, int kind, float* out, cudaStream_t stream,
                        float* theta, float lr) {
  if (theta != nullptr)
    return kind == kGaussian ? launch_grad_kind<kGaussian, true>(fitness, seeds, pop, m, offset,
                                                                 scale, out, theta, lr, stream)
                             : launch_grad_kind<kUniform, true>(fitness, seeds, pop, m, offset,
                                                                scale, out, theta, lr, stream);
  return kind == kGaussian ? launch_grad_kind<kGaussian, false>(fitness, seeds, pop, m, offset,
                                                                scale, out, nullptr, 0.f, stream)
                           : launch_grad_kind<kUniform, false>(fitness, seeds, pop, m, offset,
                                                               scale, out, nullptr, 0.f, stream);
}

}  // namespace vn
