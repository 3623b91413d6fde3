// vn_linear_ffma.cu -- the perturbed linear on CUDA cores (fp32 arithmetic).
//
// EvoX API page "evox.triton_kernels.kernels.virtual_noise", entry
// "virtual_perturbed_linear" and the module description:
//   Y[i] = X[i] @ (W + sigma*N_i)^T + (b + sigma*nb_i)
// with N_i[j,k] at offset + j*in + k and nb_i[j] at offset + out*in + j.
// The noise is "generated on-the-fly ... and added to the weight tile in
// registers" (module description): no noise tensor exists in memory.
//
// This path serves fp32 inputs and small per-individual batches (the ES
// policy case, batch 1), where there is too little reuse of each perturbed
// weight for tensor cores to matter: the work is one hash per (i, j, k) plus
// `batch` FMAs.
//
// Work decomposition: a CTA owns 32 output rows j (one per lane) for 8
// individuals (one per warp), and walks k in tiles of 64. Each tile of W is
// staged once in shared memory as W - 1.5*sigma (so that the perturbed weight
// is one FMA from the hash bits: sigma*(1+u) + W - 1.5*sigma = W + sigma*n)
// and serves all 8 individuals; each individual's X tile is staged next to it
// and read back as 16-byte broadcasts. A thread walks its row's elements in
// order, so each next state is the previous plus GAMMA. Batches larger than
// the register budget (8 rows) are done 8 rows at a time, hashing again.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "vn_hash.cuh"
#include "vn_internal.h"

namespace vn {
namespace {

constexpr int kRows = 32;   // output rows per CTA (lanes)
constexpr int kInds = 8;    // individuals per CTA (warps)
constexpr int kThreads = kRows * kInds;
constexpr int kKT = 64;     // k tile
constexpr int kWStride = kKT + 4;  // conflict-free 16-byte row reads

template <bool kBf16>
__device__ __forceinline__ float load_elem(const void* p, int64_t idx) {
  if constexpr (kBf16) {
    return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(p)[idx]);
  } else {
    return reinterpret_cast<const float*>(p)[idx];
  }
}

template <int NB, bool kXBf16, bool kWBf16>
__global__ void __launch_bounds__(kThreads)
linear_ffma_kernel(const LinearArgs a, int64_t row_tiles, int64_t tiles) {
  extern __shared__ float4 smem4[];
  float* s_w = reinterpret_cast<float*>(smem4);  // [kRows][kWStride]
  float* s_x = s_w + kRows * kWStride;           // [slabs][NB][kKT]

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int slabs = a.x_shared ? 1 : kInds;
  const float sigma = a.sigma;
  const float shift = -1.5f * sigma;

  for (int64_t t = blockIdx.x; t < tiles; t += gridDim.x) {
    const int64_t it = t / row_tiles;
    const int64_t i0 = it * kInds;
    const int64_t j0 = (t - it * row_tiles) * kRows;
    const int64_t i = i0 + warp;
    const int64_t j = j0 + lane;
    const bool live = (i < a.pop) && (j < a.out);
    const uint64_t seed = (i < a.pop) ? static_cast<uint64_t>(a.seeds[i]) : 0ull;

    for (int64_t r0 = 0; r0 < a.batch; r0 += NB) {
      float acc[NB];
#pragma unroll
      for (int r = 0; r < NB; ++r) acc[r] = 0.f;
      uint32_t slo, shi;
      index_term(a.offset + static_cast<uint64_t>(j) * static_cast<uint64_t>(a.in), slo, shi);
      add64(slo, shi, static_cast<uint32_t>(seed), static_cast<uint32_t>(seed >> 32));

      for (int64_t k0 = 0; k0 < a.in; k0 += kKT) {
        __syncthreads();  // previous tile fully consumed
        for (int q = threadIdx.x; q < kRows * kKT; q += kThreads) {
          const int rr = q / kKT, cc = q % kKT;
          const int64_t jj = j0 + rr, kk = k0 + cc;
          float v = 0.f;
          if (jj < a.out && kk < a.in) v = load_elem<kWBf16>(a.w, jj * a.in + kk) + shift;
          s_w[rr * kWStride + cc] = v;
        }
        for (int q = threadIdx.x; q < slabs * NB * kKT; q += kThreads) {
          const int s = q / (NB * kKT);
          const int rem = q % (NB * kKT);
          const int r = rem / kKT, cc = rem % kKT;
          const int64_t ii = i0 + s, rr = r0 + r, kk = k0 + cc;
          float v = 0.f;
          if ((a.x_shared || ii < a.pop) && rr < a.batch && kk < a.in) {
            const int64_t base = a.x_shared ? 0 : ii * a.batch * a.in;
            v = load_elem<kXBf16>(a.x, base + rr * a.in + kk);
          }
          s_x[q] = v;
        }
        __syncthreads();
        if (live) {
          const float* wrow = s_w + lane * kWStride;
          const float* xs = s_x + (a.x_shared ? 0 : warp) * NB * kKT;
#pragma unroll 2
          for (int kk = 0; kk < kKT; kk += 4) {
            const float4 wm = *reinterpret_cast<const float4*>(wrow + kk);
            float wp[4];
            wp[0] = fmaf(sigma, __uint_as_float(mix_to_one_plus_u(slo, shi)), wm.x);
            add64(slo, shi, kGammaLo, kGammaHi);
            wp[1] = fmaf(sigma, __uint_as_float(mix_to_one_plus_u(slo, shi)), wm.y);
            add64(slo, shi, kGammaLo, kGammaHi);
            wp[2] = fmaf(sigma, __uint_as_float(mix_to_one_plus_u(slo, shi)), wm.z);
            add64(slo, shi, kGammaLo, kGammaHi);
            wp[3] = fmaf(sigma, __uint_as_float(mix_to_one_plus_u(slo, shi)), wm.w);
            add64(slo, shi, kGammaLo, kGammaHi);
#pragma unroll
            for (int r = 0; r < NB; ++r) {
              const float4 xv = *reinterpret_cast<const float4*>(xs + r * kKT + kk);
              acc[r] = fmaf(xv.x, wp[0], acc[r]);
              acc[r] = fmaf(xv.y, wp[1], acc[r]);
              acc[r] = fmaf(xv.z, wp[2], acc[r]);
              acc[r] = fmaf(xv.w, wp[3], acc[r]);
            }
          }
        }
      }

      if (live) {
        float bias = 0.f;
        if (a.b != nullptr) {
          const float bj = (a.b_dt == VN_BF16)
                               ? __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(a.b)[j])
                               : reinterpret_cast<const float*>(a.b)[j];
          const uint64_t bidx = a.offset + static_cast<uint64_t>(a.out) * static_cast<uint64_t>(a.in) +
                                static_cast<uint64_t>(j);
          bias = fmaf(sigma, noise_at(seed, bidx), bj);
        }
#pragma unroll
        for (int r = 0; r < NB; ++r) {
          const int64_t rr = r0 + r;
          if (rr < a.batch) {
            float v = acc[r] + bias;
            if (a.act == VN_ACT_TANH) v = tanhf(v);
            const int64_t o = (i * a.batch + rr) * a.out + j;
            if (a.y_dt == VN_BF16)
              reinterpret_cast<__nv_bfloat16*>(a.y)[o] = __float2bfloat16_rn(v);
            else
              reinterpret_cast<float*>(a.y)[o] = v;
          }
        }
      }
    }
  }
}

template <int NB, bool kX, bool kW>
cudaError_t launch_nb(const LinearArgs& a, cudaStream_t stream, int sm_count) {
  const int64_t row_tiles = (a.out + kRows - 1) / kRows;
  const int64_t ind_tiles = (a.pop + kInds - 1) / kInds;
  const int64_t tiles = row_tiles * ind_tiles;
  const int slabs = a.x_shared ? 1 : kInds;
  const size_t smem = sizeof(float) * (kRows * kWStride + slabs * NB * kKT);
  auto fn = linear_ffma_kernel<NB, kX, kW>;
  static int occ = 0;
  if (occ == 0 &&
      (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, fn, kThreads, sizeof(float) * (kRows * kWStride + kInds * NB * kKT)) != cudaSuccess ||
       occ < 1))
    occ = 1;
  const int64_t grid = std::min<int64_t>(tiles, static_cast<int64_t>(sm_count) * occ * 4);
  fn<<<static_cast<unsigned>(grid), kThreads, smem, stream>>>(a, row_tiles, tiles);
  return cudaGetLastError();
}

template <bool kX, bool kW>
cudaError_t launch_dt(const LinearArgs& a, cudaStream_t stream, int sm_count) {
  if (a.batch <= 1) return launch_nb<1, kX, kW>(a, stream, sm_count);
  if (a.batch <= 2) return launch_nb<2, kX, kW>(a, stream, sm_count);
  if (a.batch <= 4) return launch_nb<4, kX, kW>(a, stream, sm_count);
  return launch_nb<8, kX, kW>(a, stream, sm_count);
}

}  // namespace

cudaError_t launch_linear_ffma(const LinearArgs& a, cudaStream_t stream) {
  DeviceInfo dev;
  cudaError_t err = device_info(&dev);
  if (err != cudaSuccess) return err;
  const bool xb = a.x_dt == VN_BF16, wb = a.w_dt == VN_BF16;
  if (xb && wb) return launch_dt<true, true>(a, stream, dev.sm_count);
  if (xb) return launch_dt<true, false>(a, stream, dev.sm_count);
  if (wb) return launch_dt<false, true>(a, stream, dev.sm_count);
  return launch_dt<false, false>(a, stream, dev.sm_count);
}

}  // namespace vn
