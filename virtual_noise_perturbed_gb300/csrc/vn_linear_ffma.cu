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
// policy case, batch 1), where each perturbed weight is used by only a few
// rows of X and the work is one hash per (i, j, k) plus `batch` FMAs.
//
// Work decomposition: a warp task is (individual i, block of up to 8 output
// rows). The lanes split one row's k range in chunks of 8 consecutive
// elements (L lanes per row, 32/L rows side by side), so each lane walks its
// chunk with the state of the next element = previous + GAMMA, reads W and
// X[i] as 16-byte vectors, and the row's partial sums meet in a warp-shuffle
// reduction. Tasks are ordered row-block-major, so the 8 warps of a CTA share
// W rows through L1, and handed out in a grid-stride loop of many small tasks,
// which keeps the last wave short. Batches above 8 rows are done 8 rows at a
// time, hashing again.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "vn_hash.cuh"
#include "vn_internal.h"

namespace vn {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kRowsPerTask = 8;

template <bool kBf16>
__device__ __forceinline__ void load8(const void* base, int64_t idx, int64_t valid, bool vec,
                                      float (&v)[8]) {
  if (vec && valid >= 8) {
    if constexpr (kBf16) {
      const uint4 r = __ldg(reinterpret_cast<const uint4*>(
          reinterpret_cast<const __nv_bfloat16*>(base) + idx));
      const uint32_t wr[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        v[2 * e] = __uint_as_float(wr[e] << 16);
        v[2 * e + 1] = __uint_as_float(wr[e] & 0xFFFF0000u);
      }
    } else {
      const float4* p = reinterpret_cast<const float4*>(reinterpret_cast<const float*>(base) + idx);
      const float4 a = __ldg(p), b = __ldg(p + 1);
      v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
      v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    }
  } else {
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      if (e < valid) {
        v[e] = kBf16 ? __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(base)[idx + e])
                     : reinterpret_cast<const float*>(base)[idx + e];
      } else {
        v[e] = 0.f;
      }
    }
  }
}

// lanes_log2: log2(L), L = lanes per output row (1..32).
template <int NB, bool kXBf16, bool kWBf16>
__global__ void __launch_bounds__(kThreads)
linear_rows_kernel(const LinearArgs a, int lanes_log2, int64_t row_blocks, int64_t tasks,
                   int x_vec, int w_vec) {
  const int lane = threadIdx.x & 31;
  const int L = 1 << lanes_log2;
  const int kl = lane & (L - 1);         // this lane's position along k
  const int rsub = lane >> lanes_log2;   // which of the warp's rows
  const int rows_per_iter = 32 >> lanes_log2;
  const int64_t kstep = static_cast<int64_t>(L) * 8;
  const float sigma = a.sigma;
  const float shift = -1.5f * sigma;
  const uint64_t bias_base = a.offset + static_cast<uint64_t>(a.out) * static_cast<uint64_t>(a.in);
  const int64_t warps_total = static_cast<int64_t>(gridDim.x) * kWarps;

  for (int64_t task = static_cast<int64_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5); task < tasks;
       task += warps_total) {
    const int64_t rb = task / a.pop;
    const int64_t i = task - rb * a.pop;
    const uint64_t seed = static_cast<uint64_t>(__ldg(a.seeds + i));
    const int64_t j_end = min(a.out, (rb + 1) * kRowsPerTask);
    for (int64_t jr = rb * kRowsPerTask; jr < j_end; jr += rows_per_iter) {
      const int64_t j = jr + rsub;
      const bool jok = j < j_end;
      for (int64_t r0 = 0; r0 < a.batch; r0 += NB) {
        float acc[NB];
#pragma unroll
        for (int r = 0; r < NB; ++r) acc[r] = 0.f;
        if (jok) {
          for (int64_t k = static_cast<int64_t>(kl) * 8; k < a.in; k += kstep) {
            const int64_t valid = a.in - k;
            float w[8];
            load8<kWBf16>(a.w, j * a.in + k, valid, w_vec != 0, w);
            uint32_t lo, hi;
            index_term(a.offset + static_cast<uint64_t>(j) * static_cast<uint64_t>(a.in) +
                           static_cast<uint64_t>(k),
                       lo, hi);
            add64(lo, hi, static_cast<uint32_t>(seed), static_cast<uint32_t>(seed >> 32));
            float wp[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              wp[e] = fmaf(sigma, __uint_as_float(mix_to_one_plus_u(lo, hi)), w[e] + shift);
              add64(lo, hi, kGammaLo, kGammaHi);
            }
#pragma unroll
            for (int r = 0; r < NB; ++r) {
              if (r0 + r < a.batch) {
                const int64_t xrow = (a.x_shared ? 0 : i * a.batch) + r0 + r;
                float x[8];
                load8<kXBf16>(a.x, xrow * a.in + k, valid, x_vec != 0, x);
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[r] = fmaf(x[e], wp[e], acc[r]);
              }
            }
          }
        }
        // Reduce over the L lanes of each row (lanes of a row are contiguous).
#pragma unroll
        for (int r = 0; r < NB; ++r) {
          for (int s = L >> 1; s > 0; s >>= 1) acc[r] += __shfl_xor_sync(0xffffffffu, acc[r], s);
        }
        if (jok && kl == 0) {
          float bias = 0.f;
          if (a.b != nullptr) {
            const float bj = (a.b_dt == VN_BF16)
                                 ? __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(a.b)[j])
                                 : reinterpret_cast<const float*>(a.b)[j];
            bias = fmaf(sigma, noise_at(seed, bias_base + static_cast<uint64_t>(j)), bj);
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
}

template <int NB, bool kX, bool kW>
cudaError_t launch_nb(const LinearArgs& a, cudaStream_t stream, int sm_count) {
  // Lanes per row: enough 8-element chunks to cover `in` once, at most 32.
  int lanes_log2 = 0;
  while (lanes_log2 < 5 && (int64_t{8} << lanes_log2) < a.in) ++lanes_log2;
  const int64_t row_blocks = (a.out + kRowsPerTask - 1) / kRowsPerTask;
  const int64_t tasks = row_blocks * a.pop;
  auto fn = linear_rows_kernel<NB, kX, kW>;
  static int occ = 0;
  if (occ == 0 &&
      (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, fn, kThreads, 0) != cudaSuccess || occ < 1))
    occ = 1;
  const int64_t grid = std::max<int64_t>(
      1, std::min<int64_t>((tasks + kWarps - 1) / kWarps, static_cast<int64_t>(sm_count) * occ));
  const size_t xe = kX ? 2 : 4, we = kW ? 2 : 4;
  const int x_vec = (a.in % (16 / xe) == 0) && (reinterpret_cast<uintptr_t>(a.x) % 16 == 0);
  const int w_vec = (a.in % (16 / we) == 0) && (reinterpret_cast<uintptr_t>(a.w) % 16 == 0);
  fn<<<static_cast<unsigned>(grid), kThreads, 0, stream>>>(a, lanes_log2, row_blocks, tasks, x_vec,
                                                            w_vec);
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
