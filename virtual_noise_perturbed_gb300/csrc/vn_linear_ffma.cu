// vn_linear_ffma.cu -- the perturbed linear on CUDA cores (fp32 arithmetic).
//
// EvoX API page "evox.triton_kernels.kernels.virtual_noise", entry
// "virtual_perturbed_linear" and the module description:
//   Y[i] = X[i] @ (W + sigma*N_i)^T + (b + sigma*nb_i)
// with N_i[j,k] at offset + j*in + k and nb_i[j] at offset + out*in + j.
// As the module description has it, the noise is made where it is used and
// added to the weights in registers: no noise tensor exists in memory.
//
// This path serves small per-individual batches with bf16 W (or bias), batches
// of 9 to 15, populations smaller than the SM count, and every call that forces
// it; layers with fp32 W of larger populations with batches up to 8 go to the
// chain kernel (vn_mlp.cu) with one layer, whose individuals share each W chunk
// a lane loads. Each
// perturbed weight meets only a few rows of X: the work is one hash per
// (i, j, k) plus `batch` FMAs.
//
// Work decomposition -- the gradient kernel's shape, turned around:
//   * A CTA owns R output rows (R = 32, or the next power of two >= out when
//     out < 32) and a contiguous slice of the population. Lane l serves row
//     l % R; the 32/R lanes of a row and the 8 warps split the row's k range
//     into 8-element chunks, up to CPT chunks per thread per k pass.
//   * A thread loads its chunks of W once, as W - 1.5*sigma in registers, with
//     the per-element part of each chunk's state, (offset + j*in + k + 1)*GAMMA.
//     It then loops over the CTA's individuals: state = that + seed, the
//     finalizer, W' = fma(sigma, 1 + u, W - 1.5*sigma) = W + sigma*n, and the
//     dot product with X[i] (staged in shared memory, read as 16-byte broadcasts).
//   * Each thread's partial sum per (individual, batch row) goes to its own
//     shared-memory slot; after the loop the partials of a row are added in a
//     fixed (warp, lane) order, then bias + bias noise + activation, and Y is
//     stored coalesced. No atomics: the result does not depend on scheduling.
//   * The number of CTAs per row tile is chosen so that the whole grid is one
//     wave of resident CTAs; a CTA's slice of the population is processed P
//     individuals at a time (P bounded by shared memory). k ranges longer than
//     one pass (8 warps x 32/R lanes x CPT chunks x 8) take several passes, and
//     batches above NB rows are done NB rows at a time, hashing again.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "vn_hash.cuh"
#include "vn_internal.h"

namespace vn {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kMaxCPT = 2;  // more chunks per thread cost more registers than they save
constexpr size_t kSmemBudget = 48 * 1024;

template <bool kBf16>
__device__ __forceinline__ float elem(const void* base, int64_t idx) {
  if constexpr (kBf16) {
    return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(base)[idx]);
  } else {
    return reinterpret_cast<const float*>(base)[idx];
  }
}

// Eight consecutive weights (fewer when `valid` < 8; the rest are 0).
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
    for (int e = 0; e < 8; ++e) v[e] = (e < valid) ? elem<kBf16>(base, idx + e) : 0.f;
  }
}

struct PopParams {
  int r_log2;         // R = 1 << r_log2 rows per CTA
  int ctas_per_tile;  // CTAs sharing one row tile (population slices)
  int p;              // individuals staged at a time
  int kpw;            // k range of one pass = 8 warps * (32/R) * CPT * 8
  int w_vec;          // W rows are 16-byte aligned for 8-element vector loads
  uint32_t g_lo, g_hi, one;  // GAMMA's halves and 1 at run time (the state step, add64_madc)
};

template <int NB, int CPT, bool kXBf16, bool kWBf16>
__global__ void __launch_bounds__(kThreads)
linear_pop_kernel(const LinearArgs a, const PopParams q) {
  extern __shared__ float4 smem4[];
  const int P = q.p;
  const int kpw = q.kpw;
  uint2* s_seed = reinterpret_cast<uint2*>(smem4);                         // [P]
  float* s_x = reinterpret_cast<float*>(smem4) + 2 * ((P + 1) & ~1);      // [P][NB][kpw]
  float* s_part = s_x + static_cast<size_t>(P) * NB * kpw;                // [8][P][NB][32]

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int R = 1 << q.r_log2;
  const int LQ = 32 >> q.r_log2;
  const int rl = lane & (R - 1);
  const int slot = (lane >> q.r_log2) + LQ * warp;  // chunk slot within a pass
  const int slots = LQ * kWarps;
  const int64_t rt = blockIdx.x / q.ctas_per_tile;
  const int64_t c = blockIdx.x - rt * q.ctas_per_tile;
  const int64_t i_begin = a.pop * c / q.ctas_per_tile;
  const int64_t i_end = a.pop * (c + 1) / q.ctas_per_tile;
  const int64_t j = rt * R + rl;
  const bool row_ok = j < a.out;
  const float sigma = a.sigma;
  const float shift = -1.5f * sigma;
  const int64_t passes = a.in > 0 ? (a.in + kpw - 1) / kpw : 1;

  for (int64_t r0 = 0; r0 < a.batch; r0 += NB) {
    for (int64_t ib = i_begin; ib < i_end; ib += P) {
      const int np = static_cast<int>(min(static_cast<int64_t>(P), i_end - ib));
      for (int64_t pass = 0; pass < passes; ++pass) {
        const int64_t kp0 = pass * kpw;
        __syncthreads();  // the previous pass / batch is done with s_x and s_seed
        for (int t = threadIdx.x; t < np; t += kThreads) {
          const uint64_t s = static_cast<uint64_t>(a.seeds[ib + t]);
          s_seed[t] = make_uint2(static_cast<uint32_t>(s), static_cast<uint32_t>(s >> 32));
        }
        const int per_ind = NB * kpw;
        for (int t = threadIdx.x; t < np * per_ind; t += kThreads) {
          const int ii = t / per_ind;
          const int rem = t - ii * per_ind;
          const int r = rem / kpw;
          const int kk = rem - r * kpw;
          const int64_t k = kp0 + kk, rr = r0 + r;
          float v = 0.f;
          if (rr < a.batch && k < a.in) {
            const int64_t row = (a.x_shared ? 0 : (ib + ii) * a.batch) + rr;
            v = elem<kXBf16>(a.x, row * a.in + k);
          }
          s_x[t] = v;
        }
        __syncthreads();

        // This thread's chunks of W for the pass, and their state terms.
        float wm[CPT][8];
        uint64_t bst[CPT];
        float sg[CPT];  // sigma for a chunk inside the pass, 0 for one past it
#pragma unroll
        for (int cq = 0; cq < CPT; ++cq) {
          const int kk = 8 * (slot + slots * cq);
          const int64_t k = kp0 + kk;
          sg[cq] = (kk < kpw) ? sigma : 0.f;
          if (row_ok && kk < kpw && k < a.in) {
            float w[8];
            load8<kWBf16>(a.w, j * a.in + k, a.in - k, q.w_vec != 0, w);
#pragma unroll
            for (int e = 0; e < 8; ++e) wm[cq][e] = w[e] + shift;
            bst[cq] = index_term(a.offset + static_cast<uint64_t>(j) * static_cast<uint64_t>(a.in) +
                                 static_cast<uint64_t>(k));
          } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) wm[cq][e] = 0.f;
            bst[cq] = 0ull;
          }
        }

        for (int ii = 0; ii < np; ++ii) {
          const uint2 sd = s_seed[ii];
          const uint64_t seed = (static_cast<uint64_t>(sd.y) << 32) | sd.x;
          float part[NB];
#pragma unroll
          for (int r = 0; r < NB; ++r) part[r] = 0.f;
          // All CPT chunks are hashed, without branches: past the end of the row
          // (k >= in) X is zero in shared memory, and a chunk past the end of the
          // pass has W' = 0 (sigma and W both 0) and reads in-bounds X.
          const float* xi = s_x + ii * NB * kpw;
#pragma unroll
          for (int cq = 0; cq < CPT; ++cq) {
            {
              const int kk = min(8 * (slot + slots * cq), kpw - 8);
              const uint64_t st = bst[cq] + seed;
              uint32_t slo = static_cast<uint32_t>(st), shi = static_cast<uint32_t>(st >> 32);
              float wp[8];
#pragma unroll
              for (int e = 0; e < 8; ++e) {
                wp[e] = fmaf(sg[cq], __uint_as_float(mix_to_one_plus_u(slo, shi)), wm[cq][e]);
                add64_madc(slo, shi, q.g_lo, q.g_hi, q.one);
              }
#pragma unroll
              for (int r = 0; r < NB; ++r) {
                const float4* xs = reinterpret_cast<const float4*>(xi + r * kpw + kk);
                const float4 xa = xs[0], xb = xs[1];
                part[r] = fmaf(xa.x, wp[0], part[r]);
                part[r] = fmaf(xa.y, wp[1], part[r]);
                part[r] = fmaf(xa.z, wp[2], part[r]);
                part[r] = fmaf(xa.w, wp[3], part[r]);
                part[r] = fmaf(xb.x, wp[4], part[r]);
                part[r] = fmaf(xb.y, wp[5], part[r]);
                part[r] = fmaf(xb.z, wp[6], part[r]);
                part[r] = fmaf(xb.w, wp[7], part[r]);
              }
            }
          }
#pragma unroll
          for (int r = 0; r < NB; ++r) {
            float* dst = s_part + ((static_cast<size_t>(warp) * P + ii) * NB + r) * 32 + lane;
            *dst = (pass == 0) ? part[r] : *dst + part[r];
          }
        }
      }
      __syncthreads();

      // Epilogue: add each row's partials in (warp, lane) order, then the bias.
      const uint64_t bias_base =
          a.offset + static_cast<uint64_t>(a.out) * static_cast<uint64_t>(a.in);
      for (int t = threadIdx.x; t < np * NB * R; t += kThreads) {
        const int ii = t / (NB * R);
        const int rem = t - ii * NB * R;
        const int r = rem / R;
        const int rr_l = rem - r * R;
        const int64_t jj = rt * R + rr_l;
        const int64_t rr = r0 + r;
        if (jj < a.out && rr < a.batch) {
          float sum = 0.f;
          for (int w = 0; w < kWarps; ++w) {
            const float* src = s_part + ((static_cast<size_t>(w) * P + ii) * NB + r) * 32;
            for (int l2 = 0; l2 < LQ; ++l2) sum += src[rr_l + l2 * R];
          }
          float bias = 0.f;
          if (a.b != nullptr) {
            const uint2 sd = s_seed[ii];
            const uint64_t seed = (static_cast<uint64_t>(sd.y) << 32) | sd.x;
            const float bj = (a.b_dt == VN_BF16)
                                 ? __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(a.b)[jj])
                                 : reinterpret_cast<const float*>(a.b)[jj];
            bias = fmaf(sigma, noise_at(seed, bias_base + static_cast<uint64_t>(jj)), bj);
          }
          float v = sum + bias;
          if (a.act == VN_ACT_TANH) v = tanhf(v);
          const int64_t o = ((ib + ii) * a.batch + rr) * a.out + jj;
          if (a.y_dt == VN_BF16)
            reinterpret_cast<__nv_bfloat16*>(a.y)[o] = __float2bfloat16_rn(v);
          else
            reinterpret_cast<float*>(a.y)[o] = v;
        }
      }
    }
  }
}

size_t smem_bytes(int p, int nb, int kpw) {
  return sizeof(float) * (2 * ((p + 1) & ~1) + static_cast<size_t>(p) * nb * kpw +
                          static_cast<size_t>(kWarps) * p * nb * 32);
}

template <int NB, int CPT, bool kX, bool kW>
cudaError_t launch_cfg(const LinearArgs& a, cudaStream_t stream, int sm_count, int r_log2) {
  auto fn = linear_pop_kernel<NB, CPT, kX, kW>;
  const int R = 1 << r_log2;
  const int LQ = 32 >> r_log2;
  PopParams q;
  q.r_log2 = r_log2;
  q.g_lo = kGammaLo;
  q.g_hi = kGammaHi;
  q.one = 1u;
  // One pass covers kWarps * LQ * CPT chunks of 8; when `in` is shorter, only
  // its (8-rounded) length is staged.
  q.kpw = static_cast<int>(std::min<int64_t>(kWarps * LQ * CPT * 8,
                                             std::max<int64_t>(8, (a.in + 7) / 8 * 8)));
  const int64_t row_tiles = (a.out + R - 1) / R;
  // P: as many individuals as the shared-memory budget allows (at most 32);
  // a single individual may need more than the default 48 KB (opt-in).
  int p = 32;
  while (p > 1 && smem_bytes(p, NB, q.kpw) > kSmemBudget) --p;
  const size_t smem = smem_bytes(p, NB, q.kpw);
  if (smem > kSmemBudget) {
    cudaError_t err =
        cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (err != cudaSuccess) return err;
  }
  int occ = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, fn, kThreads, smem) != cudaSuccess ||
      occ < 1)
    occ = 1;
  const int64_t resident = static_cast<int64_t>(sm_count) * occ;
  // One wave: split each row tile's population over resident / row_tiles CTAs.
  const int64_t per_tile = std::max<int64_t>(1, std::min<int64_t>(a.pop, resident / row_tiles));
  q.ctas_per_tile = static_cast<int>(per_tile);
  q.p = static_cast<int>(std::min<int64_t>(p, (a.pop + per_tile - 1) / per_tile));
  const size_t we = kW ? 2 : 4;
  q.w_vec = (a.in % (16 / we) == 0) && (reinterpret_cast<uintptr_t>(a.w) % 16 == 0);
  const int64_t grid = row_tiles * per_tile;
  fn<<<static_cast<unsigned>(grid), kThreads, smem_bytes(q.p, NB, q.kpw), stream>>>(a, q);
  return cudaGetLastError();
}

template <int NB, bool kX, bool kW>
cudaError_t launch_nb(const LinearArgs& a, cudaStream_t stream, int sm_count) {
  int r_log2 = 0;
  while (r_log2 < 5 && (int64_t{1} << r_log2) < a.out) ++r_log2;
  const int64_t slots = static_cast<int64_t>(kWarps) * (32 >> r_log2);
  const int64_t chunks = (a.in + 7) / 8;
  const int64_t cpt = std::max<int64_t>(1, (chunks + slots - 1) / slots);
  if (cpt <= 1) return launch_cfg<NB, 1, kX, kW>(a, stream, sm_count, r_log2);
  return launch_cfg<NB, kMaxCPT, kX, kW>(a, stream, sm_count, r_log2);
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
