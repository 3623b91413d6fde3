// vn_hash.cuh -- the splitmix64 noise core, on 32-bit halves.
//
// Definition (EvoX API page "evox.triton_kernels.kernels.virtual_noise",
// entries "_SPLITMIX64_GAMMA", "_splitmix64_step", "_cpu_normal_noise" and
// section "Noise indexing scheme"):
//   state = seed + (idx + 1) * GAMMA                         mod 2^64
//   z = (state ^ (state >> 30)) * GAMMA; z = (z ^ (z >> 27)) * GAMMA; z ^= z >> 31
//   noise = (lo32(z) >> 9) * 2^-23 - 0.5
// The state formula is this library's reading (the page leaves the mixing of
// seed and index open): the idx-th output of a splitmix64 generator.
//
// The GPU has no 64-bit integer ALU, so every 64-bit step is written on
// (hi, lo) 32-bit halves:
//   * a logical right shift of the pair is a funnel shift (low word) plus a
//     plain shift (high word);
//   * the product by GAMMA mod 2^64 is one 32x32->64 multiply of the low words
//     plus two 32-bit multiply-adds for the cross terms (GAMMA_hi*lo and
//     GAMMA_lo*hi); the hi*hi term falls off the top;
//   * only the low 32 bits of the final "z ^= z >> 31" are needed, and only
//     their top 23 bits: bits 9..31 of lo ^ (lo >> 31 | hi << 1) equal
//     (lo >> 9) ^ ((hi >> 8) & 0x7FFFFF). OR-ing in the exponent of 1.0f
//     (0x3F800000, bits 23..29) also overwrites bit 23, so the mask is free:
//     bits = ((lo >> 9) ^ (hi >> 8)) | 0x3F800000 is the float 1 + u, u in [0,1).
//   * 1 + u - 1.5 is exact in fp32, so the noise value is exact.
#pragma once

#include <cstdint>

namespace vn {

constexpr uint32_t kGammaLo = 0x7F4A7C15u;
constexpr uint32_t kGammaHi = 0x9E3779B9u;
constexpr uint64_t kGamma = 0x9E3779B97F4A7C15ull;
constexpr uint32_t kOneBits = 0x3F800000u;  // 1.0f

// 64-bit add on halves with an explicit carry chain (two integer ops).
__device__ __forceinline__ void add64(uint32_t& lo, uint32_t& hi, uint32_t alo, uint32_t ahi) {
  asm("add.cc.u32 %0, %0, %2;\n\taddc.u32 %1, %1, %3;"
      : "+r"(lo), "+r"(hi)
      : "r"(alo), "r"(ahi));
}

// The same add with the high word as a multiply-add by `one` (a run-time 1
// that the compiler cannot fold): the carry half then issues on the IMAD pipe
// instead of the integer ALU, which the finalizer already keeps the busiest.
// `one` must come from a kernel argument, not a literal.
__device__ __forceinline__ void add64_madc(uint32_t& lo, uint32_t& hi, uint32_t alo, uint32_t ahi,
                                           uint32_t one) {
  asm("add.cc.u32 %0, %0, %2;\n\tmadc.lo.u32 %1, %1, %4, %3;"
      : "+r"(lo), "+r"(hi)
      : "r"(alo), "r"(ahi), "r"(one));
}

// (hi:lo) * GAMMA mod 2^64, on halves.
__device__ __forceinline__ void mul_gamma(uint32_t lo, uint32_t hi, uint32_t& rlo, uint32_t& rhi) {
  const uint64_t p = static_cast<uint64_t>(lo) * kGammaLo;  // 32x32 -> 64
  rlo = static_cast<uint32_t>(p);
  rhi = static_cast<uint32_t>(p >> 32) + lo * kGammaHi + hi * kGammaLo;
}

// The finalizer applied to the state (hi:lo); returns the fp32 bit pattern of
// 1 + u, where u = (lo32(z) >> 9) * 2^-23.
__device__ __forceinline__ uint32_t mix_to_one_plus_u(uint32_t lo, uint32_t hi) {
  // z ^= z >> 30
  const uint32_t l1 = lo ^ __funnelshift_r(lo, hi, 30);
  const uint32_t h1 = hi ^ (hi >> 30);
  // z *= GAMMA
  uint32_t l2, h2;
  mul_gamma(l1, h1, l2, h2);
  // z ^= z >> 27
  const uint32_t l3 = l2 ^ __funnelshift_r(l2, h2, 27);
  const uint32_t h3 = h2 ^ (h2 >> 27);
  // z *= GAMMA
  uint32_t l4, h4;
  mul_gamma(l3, h3, l4, h4);
  // z ^= z >> 31, low 32 bits, top 23 of them, as the mantissa of 1.0f
  return ((l4 >> 9) ^ (h4 >> 8)) | kOneBits;
}

// The same on a 64-bit state (plain 64-bit adds on the state compile to a
// carry pair that the compiler schedules better than hand-written ones).
__device__ __forceinline__ uint32_t mix_to_one_plus_u(uint64_t state) {
  return mix_to_one_plus_u(static_cast<uint32_t>(state), static_cast<uint32_t>(state >> 32));
}

// Bits from mix_to_one_plus_u -> the noise value (1 + u) - 1.5, exact.
__device__ __forceinline__ float noise_from_bits(uint32_t bits) {
  return __uint_as_float(bits) - 1.5f;
}

// (idx + 1) * GAMMA mod 2^64: the per-element part of the state.
__device__ __forceinline__ uint64_t index_term(uint64_t idx) { return (idx + 1ull) * kGamma; }

// (idx + 1) * GAMMA mod 2^64 as halves: the per-element part of the state.
__device__ __forceinline__ void index_term(uint64_t idx, uint32_t& lo, uint32_t& hi) {
  const uint64_t t = (idx + 1ull) * kGamma;
  lo = static_cast<uint32_t>(t);
  hi = static_cast<uint32_t>(t >> 32);
}

// The full 64-bit finalizer output (zhi:zlo) of the state (hi:lo).
__device__ __forceinline__ void mix64_halves(uint32_t lo, uint32_t hi, uint32_t& zlo,
                                             uint32_t& zhi) {
  const uint32_t l1 = lo ^ __funnelshift_r(lo, hi, 30);
  const uint32_t h1 = hi ^ (hi >> 30);
  uint32_t l2, h2;
  mul_gamma(l1, h1, l2, h2);
  const uint32_t l3 = l2 ^ __funnelshift_r(l2, h2, 27);
  const uint32_t h3 = h2 ^ (h2 >> 27);
  uint32_t l4, h4;
  mul_gamma(l3, h3, l4, h4);
  zlo = l4 ^ __funnelshift_r(l4, h4, 31);
  zhi = h4 ^ (h4 >> 31);
}

// Gaussian variant: Box-Muller on the two halves of one finalizer output,
//   u1 = 1 - (zhi >> 9) 2^-23 in (0, 1],  u2 = (zlo >> 9) 2^-23 in [0, 1),
//   G = sqrt(-2 ln u1) cos(2 pi u2)
//     = kGaussScale * sqrt(-log2 u1) * cos(2 pi (u2 - 1/2)),  kGaussScale = -sqrt(2 ln 2).
// gaussian_unit() returns the last two factors; callers apply kGaussScale (the
// gradient folds it into the fitness weight). Both uniforms are formed exactly
// through the mantissa of 1.0f; log2, the reciprocal square root and cos (on
// [-pi, pi)) are the hardware approximations, whose error bounds give
// |G - exact| <= 6e-4 where u1 is within ~2^-12 of 1 (G near 0) and about 1e-6
// elsewhere.
// The three approximations are the PTX .approx.ftz instructions: every operand
// here is either 0 or a normal number (u1 >= 2^-23, m + 1e-30 >= 1e-30), so flushing
// subnormals changes nothing and saves the subnormal checks.
constexpr float kGaussScale = -1.17741002f;
__device__ __forceinline__ float lg2_approx(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float rsqrt_approx(float x) {
  float y;
  asm("rsqrt.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float cos_approx(float x) {
  float y;
  asm("cos.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float gaussian_unit(uint32_t zlo, uint32_t zhi) {
  const float u1 = 2.0f - __uint_as_float((zhi >> 9) | kOneBits);
  const float a = __uint_as_float((zlo >> 9) | kOneBits) - 1.5f;  // u2 - 1/2 in [-1/2, 1/2)
  const float m = -lg2_approx(u1);                               // -log2 u1 >= 0
  // sqrt(m) as m * rsqrt(m + 1e-30): exact 0 for m = 0 (u1 = 1), and the added
  // 1e-30 vanishes in the rounding for every other m (m >= 1.7e-7).
  return m * rsqrt_approx(m + 1e-30f) * cos_approx(6.28318531f * a);
}

// The noise value of the state (hi:lo) for either kind (the Gaussian one
// without kGaussScale: see gaussian_unit).
enum NoiseKind { kUniform = 0, kGaussian = 1 };
template <int kKind>
__device__ __forceinline__ float noise_value(uint32_t lo, uint32_t hi) {
  if constexpr (kKind == kGaussian) {
    uint32_t zlo, zhi;
    mix64_halves(lo, hi, zlo, zhi);
    return gaussian_unit(zlo, zhi);
  } else {
    return __uint_as_float(mix_to_one_plus_u(lo, hi)) - 1.5f;
  }
}

// The noise value of element idx of individual seed for either kind, the
// Gaussian one with kGaussScale applied (used where the cost does not matter).
template <int kKind>
__device__ __forceinline__ float noise_at_kind(uint64_t seed, uint64_t idx) {
  const uint64_t s = seed + (idx + 1ull) * kGamma;
  const float v = noise_value<kKind>(static_cast<uint32_t>(s), static_cast<uint32_t>(s >> 32));
  return kKind == kGaussian ? kGaussScale * v : v;
}

// PRNG(seed, idx) in one call (used where the cost does not matter).
__device__ __forceinline__ float noise_at(uint64_t seed, uint64_t idx) {
  const uint64_t s = seed + (idx + 1ull) * kGamma;
  return noise_from_bits(
      mix_to_one_plus_u(static_cast<uint32_t>(s), static_cast<uint32_t>(s >> 32)));
}

}  // namespace vn
