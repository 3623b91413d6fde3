// vn_mlp.cu -- a chain of perturbed linear layers (an ES policy) in one launch.
//
// EvoX API page "evox.triton_kernels.kernels.virtual_noise": each layer is the
// "virtual_perturbed_linear" entry,
//   h_{l+1}[i] = act_l( h_l[i] @ (W_l + sigma*N_{i,l})^T + (b_l + sigma*nb_{i,l}) ),
// with N_{i,l}[j,k] at offset_l + j*in_l + k and nb_{i,l}[j] at
// offset_l + out_l*in_l + j ("Noise indexing scheme"), and the layers' offsets
// laid out by "compute_offsets". The activation between layers (tanh) is not
// part of the method; the last layer has none.
//
// Why one launch: at the policy sizes (batch 1 per individual, layers of a few
// hundred units) a layer is a few microseconds of hashing, so separate
// launches pay a launch gap and a full-device drain per layer, and the small
// last layer cannot fill the GPU. Here an individual's activations never leave
// shared memory: a CTA takes a group of P consecutive individuals (P =
// ceil(pop / SMs), at most 8 / batch, a compile-time constant) and runs them
// through every layer.
//
// Work of one layer inside a CTA (16 warps):
//   * A row of W_l is split into 8-element chunks; LR lanes (a power of two,
//     at most 32) share a row, each taking every LR-th chunk, so a warp covers
//     32/LR rows at a time and the warps take row groups round-robin. LR is
//     the smallest power of two that gives every thread a row slot (2 for 256
//     rows on 512 threads, 32 for 8 rows), so wide layers need only a short
//     butterfly per row and the lanes of a warp read the same activation chunk
//     (a shared-memory broadcast).
//   * Per chunk a lane loads the 8 weights once (from L2: W is shared by the
//     whole population) as W - 1.5*sigma with the chunk's state term
//     (offset + j*in + k + 1)*GAMMA, then for each of the P individuals hashes
//     the 8 elements, forms W' = fma(sigma, 1 + u, W - 1.5*sigma) = W +
//     sigma*n and adds W' . h[i][k..k+7] to that individual's partial sum. The
//     next chunk's weights are loaded while this one is hashed.
//   * The LR partials of a row are summed with an xor butterfly (fixed order,
//     deterministic); lane q of the group then finishes the (individual, batch
//     row) pairs congruent to q: bias, bias noise, activation, and the value
//     goes to the other activation buffer in shared memory.
//   * Chunks past the end of a row read zero activations (each buffer is
//     zero-padded to the length the next layer reads) and rows past `out`
//     are computed on zero weights and discarded, so no lane branches on
//     ragged edges.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "vn_hash.cuh"
#include "vn_internal.h"

namespace vn {
namespace {

constexpr int kWarps = 16;
constexpr int kThreads = kWarps * 32;
constexpr int kAcc = 8;              // accumulators per lane: individuals x batch rows per group
constexpr int kSeedFloats = 16;      // shared-memory words reserved for the group's seeds

struct MlpLayerDev {
  const float* w;
  const float* b;   // may be null
  uint64_t offset;  // weight block offset; bias noise at offset + out*in
  int in, out;
  int lr_log2;      // LR = 1 << lr_log2 lanes per row
  int cpl;          // chunks per lane: ceil(ceil(in / 8) / LR)
  int in_pad;       // length this layer reads from its input buffer: LR * cpl * 8
  int w_vec;        // W rows are 16-byte aligned and in % 8 == 0: two float4 loads per chunk
};

struct MlpDev {
  MlpLayerDev layer[kMlpMaxLayers];
  const void* x;
  const int64_t* seeds;
  float* y;
  int64_t pop;
  int batch;
  int n_layers;
  int x_shared;
  int act;       // between layers
  int act_last;  // after the last layer
  int x_bf16;   // x is bf16 (else fp32)
  int buf_len;  // floats per (individual, batch row) in an activation buffer, a multiple of 8
  float sigma;
  uint32_t g_lo, g_hi, one;  // GAMMA's halves and 1, at run time (the state step, add64_madc)
};

// Eight weights of row j from column k (zeros outside the matrix).
__device__ __forceinline__ void load_w8(const float* w, int in, int out, bool vec, int j, int k,
                                        float (&v)[8]) {
  if (j < out && k < in) {
    const float* src = w + static_cast<int64_t>(j) * in + k;
    if (vec) {
      const float4 a = __ldg(reinterpret_cast<const float4*>(src));
      const float4 b = __ldg(reinterpret_cast<const float4*>(src) + 1);
      v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
      v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) v[e] = (k + e < in) ? __ldg(src + e) : 0.f;
    }
  } else {
#pragma unroll
    for (int e = 0; e < 8; ++e) v[e] = 0.f;
  }
}

// CTA c runs individuals [c*kP, c*kP + kP) through every layer. The group size
// kP is a compile-time constant so that the kP x 8 hashes of a chunk are
// straight-line code the compiler can interleave; a CTA at the end of the
// population with fewer individuals hashes its last one again in the empty
// slots (the same wall time: the other CTAs have a full group) and stores
// nothing for them.
template <int NB, int kP, int kKind>
__global__ void __launch_bounds__(kThreads, 1) mlp_kernel(const __grid_constant__ MlpDev a) {
  extern __shared__ float4 smem4[];
  float* smem = reinterpret_cast<float*>(smem4);
  uint2* s_seed = reinterpret_cast<uint2*>(smem);                 // [kP]
  const int blen = a.buf_len;
  // Two activation buffers [kP][NB][blen], `bstride` floats apart.
  float* const s_buf0 = smem + kSeedFloats;
  const int bstride = kP * NB * blen;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const float sigma = a.sigma;
  // Uniform kind: W' = fma(sigma, 1 + u, W - 1.5*sigma). Gaussian kind: W' =
  // fma(sigma * kGaussScale, unit, W), unit = gaussian_unit of the finalizer's halves.
  const float shift = kKind == kGaussian ? 0.f : -1.5f * sigma;
  const float sigma_unit = kKind == kGaussian ? sigma * kGaussScale : sigma;
  const int64_t ib = static_cast<int64_t>(blockIdx.x) * kP;
  const int np = static_cast<int>(min(static_cast<int64_t>(kP), a.pop - ib));

  for (int t = threadIdx.x; t < kP; t += kThreads) {
    const uint64_t s = static_cast<uint64_t>(a.seeds[ib + min(t, np - 1)]);
    s_seed[t] = make_uint2(static_cast<uint32_t>(s), static_cast<uint32_t>(s >> 32));
  }
  // Stage x: zero past `in`, for batch rows >= batch and for the empty slots.
  {
    const int in0 = a.layer[0].in;
    const int per = NB * blen;
    const bool xb = a.x_bf16 != 0;
    for (int t = threadIdx.x; t < kP * per; t += kThreads) {
      const int ii = t / per;
      const int rem = t - ii * per;
      const int r = rem / blen;
      const int k = rem - r * blen;
      float v = 0.f;
      if (ii < np && r < a.batch && k < in0) {
        const int64_t row = (a.x_shared ? 0 : (ib + ii) * a.batch) + r;
        v = xb ? __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(a.x)[row * in0 + k])
               : reinterpret_cast<const float*>(a.x)[row * in0 + k];
      }
      s_buf0[t] = v;
    }
  }
  __syncthreads();

  for (int l = 0; l < a.n_layers; ++l) {
    // The layer's parameters, read once into registers.
    const float* const Lw = a.layer[l].w;
    const float* const Lb = a.layer[l].b;
    const uint64_t Loff = a.layer[l].offset;
    const int Lin = a.layer[l].in;
    const int Lout = a.layer[l].out;
    const int lr_log2 = a.layer[l].lr_log2;
    const int cpl = a.layer[l].cpl;
    const bool wvec = a.layer[l].w_vec != 0;
    const float* src = s_buf0 + (l & 1) * bstride;
    float* dst = s_buf0 + ((l & 1) ^ 1) * bstride;
    const bool last = l + 1 == a.n_layers;
    const bool tanh_act = (last ? a.act_last : a.act) == VN_ACT_TANH;
    const int LR = 1 << lr_log2;
    const int q = lane & (LR - 1);         // lane within its row group
    const int rsub = lane >> lr_log2;      // row of this lane within the warp's group
    const int rows_per_group = 32 >> lr_log2;
    const int n_rg = (Lout + rows_per_group - 1) / rows_per_group;
    const int my_rg = n_rg > warp ? (n_rg - warp + kWarps - 1) / kWarps : 0;
    const int steps = my_rg * cpl;
    const uint64_t bias_base = Loff + static_cast<uint64_t>(Lout) * static_cast<uint64_t>(Lin);

    // State term step between a lane's consecutive chunks of a row (8*LR elements).
    const uint64_t chunk_step = static_cast<uint64_t>(8 << lr_log2) * kGamma;

    float part[kP][NB];
    float wn[8];
    uint64_t bst = 0;  // (Loff + j*in + k + 1) * GAMMA of the current chunk's first element
    if (steps > 0) load_w8(Lw, Lin, Lout, wvec, warp * rows_per_group + rsub, q * 8, wn);
    for (int s = 0, rgi = 0, m = 0; s < steps; ++s) {
      const int j = (warp + rgi * kWarps) * rows_per_group + rsub;
      const int k = (q + (m << lr_log2)) * 8;
      // A row's first chunk: its state term from the index; the next ones add chunk_step.
      bst = (m == 0) ? index_term(Loff + static_cast<uint64_t>(j) * static_cast<uint64_t>(Lin) +
                                  static_cast<uint64_t>(k))
                     : bst + chunk_step;
      if (m == 0) {
#pragma unroll
        for (int ii = 0; ii < kP; ++ii)
#pragma unroll
          for (int r = 0; r < NB; ++r) part[ii][r] = 0.f;
      }
      float wm[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) wm[e] = wn[e] + shift;
      // The next step's chunk: the same row's next one, or the next row group's first.
      const int m1 = (m + 1 < cpl) ? m + 1 : 0;
      const int rgi1 = (m + 1 < cpl) ? rgi : rgi + 1;
      if (s + 1 < steps)
        load_w8(Lw, Lin, Lout, wvec, (warp + rgi1 * kWarps) * rows_per_group + rsub,
                (q + (m1 << lr_log2)) * 8, wn);
      const float* hk = src + k;
#pragma unroll
      for (int ii = 0; ii < kP; ++ii) {
        const uint2 sd = s_seed[ii];
        const uint64_t st = bst + ((static_cast<uint64_t>(sd.y) << 32) | sd.x);
        uint32_t slo = static_cast<uint32_t>(st), shi = static_cast<uint32_t>(st >> 32);
        float wp[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          if constexpr (kKind == kGaussian) {
            uint32_t zlo, zhi;
            mix64_halves(slo, shi, zlo, zhi);
            wp[e] = fmaf(sigma_unit, gaussian_unit(zlo, zhi), wm[e]);
          } else {
            wp[e] = fmaf(sigma_unit, __uint_as_float(mix_to_one_plus_u(slo, shi)), wm[e]);
          }
          add64_madc(slo, shi, a.g_lo, a.g_hi, a.one);
        }
#pragma unroll
        for (int r = 0; r < NB; ++r) {
          const float4* h = reinterpret_cast<const float4*>(hk + (ii * NB + r) * blen);
          const float4 xa = h[0], xb = h[1];
          float acc = part[ii][r];
          acc = fmaf(xa.x, wp[0], acc);
          acc = fmaf(xa.y, wp[1], acc);
          acc = fmaf(xa.z, wp[2], acc);
          acc = fmaf(xa.w, wp[3], acc);
          acc = fmaf(xb.x, wp[4], acc);
          acc = fmaf(xb.y, wp[5], acc);
          acc = fmaf(xb.z, wp[6], acc);
          acc = fmaf(xb.w, wp[7], acc);
          part[ii][r] = acc;
        }
      }
      if (m + 1 == cpl) {
        // Sum the row's LR partials (every lane of the group ends with the total).
        for (int o = LR >> 1; o > 0; o >>= 1) {
#pragma unroll
          for (int ii = 0; ii < kP; ++ii)
#pragma unroll
            for (int r = 0; r < NB; ++r)
              part[ii][r] += __shfl_xor_sync(0xffffffffu, part[ii][r], o);
        }
        // Lane q of the row's group finishes the (individual, batch row) pairs
        // pr = ii*NB + r congruent to q mod LR: bias, bias noise, activation.
        if (j < Lout) {
          const float bj = Lb != nullptr ? __ldg(Lb + j) : 0.f;
          constexpr int kPairs = kP * NB;
          for (int base = 0; base < kPairs; base += LR) {
            const int pr = base + q;
            if (pr < kPairs) {
              float v = part[0][0];
#pragma unroll
              for (int t = 1; t < kPairs; ++t)
                if (pr == t) v = part[t / NB][t % NB];
              if (Lb != nullptr) {
                const uint2 sd = s_seed[pr / NB];
                const uint64_t seed = (static_cast<uint64_t>(sd.y) << 32) | sd.x;
                v += fmaf(sigma, noise_at_kind<kKind>(seed, bias_base + static_cast<uint64_t>(j)), bj);
              }
              if (tanh_act) v = tanhf(v);
              dst[pr * blen + j] = v;
            }
          }
        }
      }
      if (++m == cpl) { m = 0; ++rgi; }
    }
    // dst must read as zeros on [out, next layer's in_pad).
    if (!last) {
      const int pad = a.layer[l + 1].in_pad - Lout;
      if (pad > 0) {
        for (int t = threadIdx.x; t < kP * NB * pad; t += kThreads) {
          const int row = t / pad;
          dst[row * blen + Lout + (t - row * pad)] = 0.f;
        }
      }
    }
    __syncthreads();
  }

  // y[i, r, j] from the last layer's buffer.
  const float* fin = s_buf0 + (a.n_layers & 1) * bstride;
  const int outl = a.layer[a.n_layers - 1].out;
  const int per = a.batch * outl;
  for (int t = threadIdx.x; t < np * per; t += kThreads) {
    const int ii = t / per;
    const int rem = t - ii * per;
    const int r = rem / outl;
    const int j = rem - r * outl;
    a.y[(ib + ii) * per + rem] = fin[(ii * NB + r) * blen + j];
  }
}

// Lanes per row (as log2), chunks per lane and the padded input length of a
// layer. Enough lanes share a row to give every thread of the CTA a row slot
// (fewer rows -> more lanes per row), but never more lanes than the row has
// chunks: the butterfly that sums a row's lanes is then short for wide layers.
struct LayerShape {
  int lr_log2, cpl, in_pad;
};
LayerShape layer_shape(int64_t in, int64_t out) {
  const int64_t chunks = std::max<int64_t>(1, (in + 7) / 8);  // in == 0: one all-zero chunk
  int lg = 0;
  while (lg < 5 && (int64_t{2} << lg) * std::max<int64_t>(out, 1) <= kThreads &&
         (int64_t{1} << lg) < chunks)
    ++lg;
  LayerShape sh;
  sh.lr_log2 = lg;
  sh.cpl = static_cast<int>((chunks + (int64_t{1} << lg) - 1) >> lg);
  sh.in_pad = sh.cpl * (8 << lg);
  return sh;
}

template <int NB, int kP, int kKind>
cudaError_t launch_p(MlpDev& d, cudaStream_t stream, size_t smem) {
  auto fn = mlp_kernel<NB, kP, kKind>;
  if (smem > 48 * 1024) {
    static SmemRecord configured;
    const cudaError_t err = ensure_dynamic_smem(reinterpret_cast<const void*>(fn), smem, configured);
    if (err != cudaSuccess) return err;
  }
  const int64_t grid = (d.pop + kP - 1) / kP;
  fn<<<static_cast<unsigned>(grid), kThreads, smem, stream>>>(d);
  return cudaGetLastError();
}

// Group size: enough individuals per CTA that one CTA per SM covers the
// population (ceil(pop / SMs)), at most kAcc / NB, and no more than the shared
// memory holds.
template <int NB, int kKind>
cudaError_t launch_nb(MlpDev& d, cudaStream_t stream, const DeviceInfo& dev) {
  constexpr int kMaxP = kAcc / NB;
  const size_t per_ind = 2ull * NB * static_cast<size_t>(d.buf_len) * sizeof(float);
  const size_t base = kSeedFloats * sizeof(float);
  const size_t budget = static_cast<size_t>(dev.smem_optin);
  if (base + per_ind > budget) return cudaErrorInvalidValue;  // checked by the caller
  int p = static_cast<int>(std::min<int64_t>(kMaxP, (d.pop + dev.sm_count - 1) / dev.sm_count));
  p = static_cast<int>(std::min<size_t>(p, (budget - base) / per_ind));
  p = std::max(p, 1);
  const size_t smem = base + static_cast<size_t>(p) * per_ind;
  if constexpr (NB == 1) {
    switch (p) {
      case 1: return launch_p<1, 1, kKind>(d, stream, smem);
      case 2: return launch_p<1, 2, kKind>(d, stream, smem);
      case 3: return launch_p<1, 3, kKind>(d, stream, smem);
      case 4: return launch_p<1, 4, kKind>(d, stream, smem);
      case 5: return launch_p<1, 5, kKind>(d, stream, smem);
      case 6: return launch_p<1, 6, kKind>(d, stream, smem);
      case 7: return launch_p<1, 7, kKind>(d, stream, smem);
      default: return launch_p<1, 8, kKind>(d, stream, smem);
    }
  } else if constexpr (NB == 2) {
    switch (p) {
      case 1: return launch_p<2, 1, kKind>(d, stream, smem);
      case 2: return launch_p<2, 2, kKind>(d, stream, smem);
      case 3: return launch_p<2, 3, kKind>(d, stream, smem);
      default: return launch_p<2, 4, kKind>(d, stream, smem);
    }
  } else if constexpr (NB == 4) {
    return p == 1 ? launch_p<4, 1, kKind>(d, stream, smem) : launch_p<4, 2, kKind>(d, stream, smem);
  } else {
    return launch_p<8, 1, kKind>(d, stream, smem);
  }
}

}  // namespace

size_t mlp_buffer_floats(int n_layers, const int64_t* dims) {
  int64_t len = 8;
  for (int l = 0; l < n_layers; ++l) {
    len = std::max<int64_t>(len, layer_shape(dims[l], dims[l + 1]).in_pad);
    len = std::max<int64_t>(len, dims[l + 1]);
  }
  return static_cast<size_t>((len + 7) / 8 * 8);
}

cudaError_t launch_mlp(const MlpArgs& m, cudaStream_t stream) {
  DeviceInfo dev;
  cudaError_t err = device_info(&dev);
  if (err != cudaSuccess) return err;
  MlpDev d{};
  for (int l = 0; l < m.n_layers; ++l) {
    MlpLayerDev& L = d.layer[l];
    L.w = m.w[l];
    L.b = m.b[l];
    L.offset = m.offsets[l];
    L.in = static_cast<int>(m.dims[l]);
    L.out = static_cast<int>(m.dims[l + 1]);
    const LayerShape sh = layer_shape(L.in, L.out);
    L.lr_log2 = sh.lr_log2;
    L.cpl = sh.cpl;
    L.in_pad = sh.in_pad;
    L.w_vec = (L.in % 8 == 0) && (reinterpret_cast<uintptr_t>(L.w) % 16 == 0);
  }
  d.x = m.x;
  d.seeds = m.seeds;
  d.y = m.y;
  d.pop = m.pop;
  d.batch = static_cast<int>(m.batch);
  d.n_layers = m.n_layers;
  d.x_shared = m.x_shared;
  d.act = m.act;
  d.act_last = m.act_last;
  d.buf_len = static_cast<int>(mlp_buffer_floats(m.n_layers, m.dims));
  d.sigma = m.sigma;
  d.g_lo = kGammaLo;
  d.g_hi = kGammaHi;
  d.one = 1u;
  d.x_bf16 = m.x_dt == VN_BF16 ? 1 : 0;
  if (m.kind == kGaussian) {
    if (m.batch <= 1) return launch_nb<1, kGaussian>(d, stream, dev);
    if (m.batch <= 2) return launch_nb<2, kGaussian>(d, stream, dev);
    if (m.batch <= 4) return launch_nb<4, kGaussian>(d, stream, dev);
    return launch_nb<8, kGaussian>(d, stream, dev);
  }
  if (m.batch <= 1) return launch_nb<1, kUniform>(d, stream, dev);
  if (m.batch <= 2) return launch_nb<2, kUniform>(d, stream, dev);
  if (m.batch <= 4) return launch_nb<4, kUniform>(d, stream, dev);
  return launch_nb<8, kUniform>(d, stream, dev);
}

}  // namespace vn
