// vn_linear_tc.cu -- the perturbed linear on 5th-generation tensor cores
// (tcgen05.mma, fp32 accumulators in TMEM, X staged by TMA).
//
// EvoX API page "evox.triton_kernels.kernels.virtual_noise", entry
// "virtual_perturbed_linear" and the module description:
//   Y[i] = X[i] @ (W + sigma*N_i)^T + (b + sigma*nb_i)
// N_i[j,k] at offset + j*in + k, nb_i[j] at offset + out*in + j. The noise is
// generated on the fly and added to the weight tile before the contraction
// (the module description adds it to the tile in registers); no noise tensor exists.
//
// Per individual the product is D = W'_i X_i^T with D[j, n] = Y_i[n, j]:
//   A = W'_i tile, 128 output rows x 64 k per swizzle atom (bf16, K-major),
//       written into shared memory by "hashing" warps in the 128-byte-swizzled
//       canonical layout from the W tile (fp32 or bf16, 128 rows x the stage's
//       64 or 128 k), which TMA stages once per (unit, k chunk) into a ring of one
//       or two slots shared by all hashing warps;
//   B = X_i tile, NT batch rows x 64 k (bf16, K-major), loaded by TMA with the
//       same 128-byte swizzle;
//   D = fp32 accumulator in TMEM, 128 lanes (output rows) x NT columns (batch).
// The contraction is tiny next to the hash work (one 64-bit splitmix64 hash per
// weight element per individual, about 20 integer operations), so the kernel is
// built around keeping the integer pipes busy:
//   warp 0      TMA producer for W and X tiles (one thread);
//   warp 1      TMEM allocator and MMA issuer (one thread);
//   warps 2..5  epilogue: TMEM -> registers -> + b + sigma*nb -> Y (one per TMEM lane quarter);
//   warps 6..21 hashing: W'_i = bf16(W + sigma*N_i), 16 bytes (8 k) per store.
// A work unit is (group of G individuals, N tile, M tile of 128*MH output rows;
// the host uses MH = 1); per k chunk (one stage: 64 k per swizzle atom, one or
// two atoms) the unit's W tile is staged once and perturbed for each of the G
// individuals, whose accumulators sit
// side by side in TMEM (G*MH*NT <= 256 columns, so two units can be in flight:
// double-buffered TMEM).
// Every barrier wait is bounded; a wait that runs out records a status word,
// makes the other roles stop, drains what was issued, frees TMEM and returns.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstring>
#include <mutex>
#include <type_traits>

#include "vn_hash.cuh"
#include "vn_internal.h"

namespace vn {

// Nonzero after a bounded wait ran out in a kernel of this file (read and
// cleared by take_device_status). Bits: 1 = barrier wait timed out.
__device__ unsigned int g_device_status = 0;

namespace {

constexpr int kHashWarps = 16;
constexpr int kFirstHashWarp = 6;
constexpr int kThreads = (kFirstHashWarp + kHashWarps) * 32;  // 704
constexpr int kHashThreads = kHashWarps * 32;                 // 512
constexpr int kAtomK = 64;                                    // k per swizzle atom (128 bytes of bf16)
constexpr uint32_t kHalfBytes = 128 * 128;                    // 128 rows x 128 bytes
constexpr int kTmemCols = 512;
constexpr unsigned long long kTimeoutNs = 4000000000ull;      // default limit of one wait: 4 s
// Back-off between polls of roles that run stages ahead of their consumers.
// The TMA producer polls without one (its waits suspend on the barrier): with
// one individual per unit every stage needs a fresh W tile, and a late copy
// stalls all hashing warps.
constexpr uint32_t kProducerSleepNs = 0;
constexpr uint32_t kMmaSleepNs = 256;
constexpr int kEpilogueFirstThread = 2 * 32;  // warps 2..5
constexpr int kEpilogueThreads = 4 * 32;
constexpr int kEpilogueBarrier = 1;           // named barrier id (0 is __syncthreads)

struct TcParams {
  const void* b;
  const int64_t* seeds;
  void* y;
  int64_t pop, batch, in, out;
  int64_t m_tiles, n_tiles, units;
  uint64_t offset;
  float sigma;
  int b_bf16, act;
  int nt, g, nbuf, stages, k_chunks, x_shared;
  uint32_t stage_bytes, a_bytes, idesc;
  uint32_t x_atom_bytes;  // one swizzle atom of the X tile: nt rows x 128 bytes
  uint32_t w_bytes;       // one W tile in shared memory: 128 rows x (64 * atoms) k of W's dtype
  int w_slots;            // W tiles in the ring (1 or 2)
  int units32;            // the unit index and its decomposition fit in 32 bits
  unsigned long long timeout_ns;  // limit of every barrier wait
  uint32_t g_lo, g_hi, one;       // GAMMA's halves and 1, passed at run time: the state
                                  // step's carry half is then a multiply-add on the IMAD
                                  // pipe (add64_madc)
  long long withhold_stage;       // test hook: >= 0 makes one thread skip that stage's arrive
};

// Shared by a CTA's roles: the abort flag (set by the first wait that runs out)
// and the limit of every wait.
struct WaitCtl {
  int abort;
  int pad;
  unsigned long long timeout_ns;
};

// ---------------------------------------------------------------- PTX helpers
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// try_wait with a suspend-time hint: a thread whose phase is not complete is
// suspended until the phase completes or `ns` nanoseconds pass, so waiting
// threads do not take issue slots from the hashing warps.
__device__ __forceinline__ bool mbar_try_wait_suspend(uint32_t bar, uint32_t parity, uint32_t ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(ns)
      : "memory");
  return ok != 0;
}
// Bounded wait on the phase with the given parity. Returns false if the wait
// ran out (the status word and the CTA's abort flag are then set) or if
// another role of the CTA has already aborted. Each poll suspends the thread
// for up to kSuspendNs (it resumes as soon as the phase completes).
constexpr uint32_t kSuspendNs = 200000;
__device__ __noinline__ bool mbar_wait_slow(uint32_t bar, uint32_t parity, volatile WaitCtl* ctl,
                                            uint32_t sleep_ns) {
  const uint64_t t0 = global_ns();
  const unsigned long long limit = ctl->timeout_ns;
  for (uint32_t n = 1;; ++n) {
    if (mbar_try_wait_suspend(bar, parity, kSuspendNs)) return true;
    if (sleep_ns) __nanosleep(sleep_ns);
    if ((n & 3) == 0) {
      if (ctl->abort) return false;
      if (global_ns() - t0 > limit) {
        atomicOr(&g_device_status, 1u);
        ctl->abort = 1;
        return false;
      }
    }
  }
}
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile WaitCtl* ctl,
                                          uint32_t sleep_ns = 0) {
  if (mbar_try_wait(bar, parity)) return true;
  return mbar_wait_slow(bar, parity, ctl, sleep_ns);
}
// Position in a ring of S slots: slot index and the parity of its current use.
struct Ring {
  int s = 0;
  uint32_t ph = 0;
  __device__ __forceinline__ void next(int n) {
    if (++s == n) {
      s = 0;
      ph ^= 1u;
    }
  }
};
// Named CTA barrier among `count` threads; may be reached by a divergent warp.
__device__ __forceinline__ void named_barrier_sync(int id, int count) {
  asm volatile("barrier.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1)
      : "memory");
}
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int c0, int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// D[tmem] (+)= A[smem] * B[smem]^T, bf16 inputs, fp32 accumulate, M=128.
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive on the mbarrier once every tcgen05 operation issued so far by this thread completes.
__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   bar)
               : "memory");
}
// 32 TMEM lanes x 16 consecutive 32-bit columns: thread t gets lane base+t.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
        "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
        "=r"(v[14]), "=r"(v[15])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}

__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle, 8-row
// groups 1024 bytes apart (stride byte offset), descriptor version 1.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr) {
  uint64_t d = static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(1) << 16;            // leading byte offset (unused for this layout)
  d |= static_cast<uint64_t>(1024 >> 4) << 32;    // stride byte offset
  d |= static_cast<uint64_t>(1) << 46;            // version
  d |= static_cast<uint64_t>(2) << 61;            // 128-byte swizzle
  return d;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// One output value, streamed to Y as bf16 (round to nearest even) or fp32.
template <bool kYBf16, typename YT>
__device__ __forceinline__ void store_y(YT* dst, float val) {
  if constexpr (kYBf16) {
    const __nv_bfloat16 hv = __float2bfloat16_rn(val);
    __stcs(dst, *reinterpret_cast<const unsigned short*>(&hv));
  } else {
    __stcs(dst, val);
  }
}

// W elements of one 16-byte output chunk (8 k): fp32 (two float4) or bf16 (one uint4).
struct RawF32 { float4 a, b; };
struct RawBf16 { uint4 a; };

// The 8 weights of a chunk as fp32, minus 1.5*sigma: sigma*(1 + u) + (W - 1.5*sigma) = W + sigma*n.
__device__ __forceinline__ void unpack_shift(const RawF32& r, float shift, float (&w)[8]) {
  w[0] = r.a.x + shift; w[1] = r.a.y + shift; w[2] = r.a.z + shift; w[3] = r.a.w + shift;
  w[4] = r.b.x + shift; w[5] = r.b.y + shift; w[6] = r.b.z + shift; w[7] = r.b.w + shift;
}

// float(bf16 half of w selected by kHi) + t, one fp32 rounding (mixed-precision add).
template <bool kHi>
__device__ __forceinline__ float add_bf16_f32(uint32_t w, float t) {
  float d;
  if constexpr (kHi) {
    asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\tadd.rn.f32.bf16 %0, hi, %2;\n\t}"
        : "=f"(d) : "r"(w), "f"(t));
  } else {
    asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\tadd.rn.f32.bf16 %0, lo, %2;\n\t}"
        : "=f"(d) : "r"(w), "f"(t));
  }
  return d;
}

// A work unit; every field fits in 32 bits on this path (pop, batch, in and out
// are below 2^31, checked on the host).
struct Unit {
  int i0;      // first individual of the group
  int gcount;  // individuals in the group
  int n0;      // first batch row
  int m0;      // first output row
};
__device__ __forceinline__ Unit decode(const TcParams& p, int64_t u, int mh) {
  Unit r;
  int64_t mt, ntile, g;
  if (p.units32) {  // 32-bit divisions: a 64-bit one is a long instruction sequence
    const uint32_t uu = static_cast<uint32_t>(u);
    const uint32_t mtiles = static_cast<uint32_t>(p.m_tiles), ntiles = static_cast<uint32_t>(p.n_tiles);
    const uint32_t rest = uu / mtiles;
    mt = uu - rest * mtiles;
    ntile = rest % ntiles;
    g = rest / ntiles;
  } else {
    mt = u % p.m_tiles;
    const int64_t rest = u / p.m_tiles;
    ntile = rest % p.n_tiles;
    g = rest / p.n_tiles;
  }
  r.i0 = static_cast<int>(g * p.g);
  r.gcount = static_cast<int>(min(static_cast<int64_t>(p.g), p.pop - r.i0));
  r.n0 = static_cast<int>(ntile * p.nt);
  r.m0 = static_cast<int>(mt * 128 * mh);
  return r;
}

// ---------------------------------------------------------------- the kernel
// kHook: the test-hook instance (one hashing thread may withhold an arrive);
// the ordinary instances carry no trace of it. kAtoms: swizzle atoms of 64 k per
// stage (K = 64 * kAtoms); two give every hashing thread 32 elements per stage,
// so each stage's waits, fences and arrivals are paid once per 32 elements.
// kFix: two stages and one W tile with an even number of k chunks per unit (one
// individual per unit): the hashing warps then address both stages and the W
// tile with compile-time offsets and carry a single parity bit.
template <int MH, bool kWBf16, bool kYBf16, bool kHook, int kKind, bool kG1, int kAtoms, bool kFix>
__global__ void __launch_bounds__(kThreads, 1)
linear_tc_kernel(const __grid_constant__ CUtensorMap xmap, const __grid_constant__ CUtensorMap wmap,
                 const TcParams p) {
  constexpr int kKC = kAtomK * kAtoms;  // k per stage
  // The fixed loop carries each chunk's state chain from one k chunk to the next
  // and takes no per-individual seed: one individual per unit only.
  static_assert(!kFix || kG1, "the fixed two-stage loop serves one individual per unit");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const int S = p.stages;
  // layout: S stages (A tile: kAtoms atoms of 128*MH rows x 128 bytes; X tile: kAtoms
  // atoms of nt rows x 128 bytes), w_slots W tiles, barriers
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + static_cast<size_t>(S) * p.stage_bytes +
                                               static_cast<size_t>(p.w_slots) * p.w_bytes);
  // barriers: full_a[S], full_x[S], empty[S], tmem_full[2], tmem_empty[2], drain,
  // full_w[2], empty_w[2]
  const uint32_t bar0 = smem_u32(bars);
  auto full_a = [&](int s) { return bar0 + 8u * s; };
  auto full_x = [&](int s) { return bar0 + 8u * (S + s); };
  auto empty = [&](int s) { return bar0 + 8u * (2 * S + s); };
  auto tmem_full = [&](int b) { return bar0 + 8u * (3 * S + b); };
  auto tmem_empty = [&](int b) { return bar0 + 8u * (3 * S + 2 + b); };
  const uint32_t drain = bar0 + 8u * (3 * S + 4);
  auto full_w = [&](int b) { return bar0 + 8u * (3 * S + 5 + b); };
  auto empty_w = [&](int b) { return bar0 + 8u * (3 * S + 7 + b); };
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(bars + 3 * S + 9);
  volatile WaitCtl* s_abort = reinterpret_cast<volatile WaitCtl*>(bars + 3 * S + 10);
  const uint32_t stage0 = smem_u32(smem);
  const uint32_t wslot0 = stage0 + S * p.stage_bytes;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full_a(s), kHashThreads);
      mbar_init(full_x(s), 1);
      mbar_init(empty(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tmem_full(b), 1);
      mbar_init(tmem_empty(b), 128);
    }
    mbar_init(drain, 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(full_w(b), 1);
      mbar_init(empty_w(b), kHashThreads);
    }
    s_abort->abort = 0;
    s_abort->timeout_ns = p.timeout_ns;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(s_tmem), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;
  const uint32_t cols_per_buf = kTmemCols / p.nbuf;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      uint32_t it = 0, wit = 0;
      Ring rg, wr;
      bool ok = true;
      const uint32_t x_bytes = p.x_atom_bytes;
      for (int64_t u = blockIdx.x; ok && u < p.units; u += gridDim.x) {
        const Unit un = decode(p, u, MH);
        for (int kc = 0; ok && kc < p.k_chunks; ++kc) {
          // The group's W tile (rows >= out and k >= in arrive as zeros).
          if (!(ok = mbar_wait(empty_w(wr.s), wr.ph ^ 1u, s_abort, kProducerSleepNs))) break;
          mbar_expect_tx(full_w(wr.s), p.w_bytes);
          tma_load_2d(wslot0 + wr.s * p.w_bytes, &wmap, full_w(wr.s), kc * kKC, un.m0);
          ++wit;
          wr.next(p.w_slots);
          for (int ii = 0; ii < (kG1 ? 1 : un.gcount); ++ii, ++it, rg.next(S)) {
            const int s = rg.s;
            if (!(ok = mbar_wait(empty(s), rg.ph ^ 1u, s_abort, kProducerSleepNs))) break;
            mbar_expect_tx(full_x(s), x_bytes * kAtoms);
            const int ind = p.x_shared ? 0 : static_cast<int>(un.i0 + ii);
#pragma unroll
            for (int a = 0; a < kAtoms; ++a)
              tma_load_3d(stage0 + s * p.stage_bytes + p.a_bytes + a * x_bytes, &xmap, full_x(s),
                          kc * kKC + a * kAtomK, static_cast<int>(un.n0), ind);
          }
        }
      }
      if (!ok) {
        // Drain: every load issued lands on its full_x barrier; wait for the
        // last S of them (bounded) so no copy is in flight at exit.
        for (uint32_t k = 0; k < static_cast<uint32_t>(S) && k < it; ++k) {
          const uint32_t j = it - 1 - k;
          const uint64_t t0 = global_ns();
          while (!mbar_try_wait(full_x(static_cast<int>(j % S)), (j / S) & 1u) &&
                 global_ns() - t0 < p.timeout_ns) {
          }
        }
        const uint32_t nw = static_cast<uint32_t>(p.w_slots);
        for (uint32_t k = 0; k < nw && k < wit; ++k) {
          const uint32_t j = wit - 1 - k;
          const uint64_t t0 = global_ns();
          while (!mbar_try_wait(full_w(static_cast<int>(j % nw)), (j / nw) & 1u) &&
                 global_ns() - t0 < p.timeout_ns) {
          }
        }
      }
    }
  } else if (warp == 1) {
    // -------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      Ring rg, tb;
      bool ok = true;
      for (int64_t u = blockIdx.x; ok && u < p.units; u += gridDim.x, tb.next(p.nbuf)) {
        const Unit un = decode(p, u, MH);
        const int b = tb.s;
        if (!(ok = mbar_wait(tmem_empty(b), tb.ph ^ 1u, s_abort, kMmaSleepNs))) break;
        tc_fence_after();
        const uint32_t dcol = tmem + b * cols_per_buf;
        for (int kc = 0; ok && kc < p.k_chunks; ++kc) {
          for (int ii = 0; ii < (kG1 ? 1 : un.gcount); ++ii, rg.next(S)) {
            const int s = rg.s;
            if (!(ok = mbar_wait(full_x(s), rg.ph, s_abort, kMmaSleepNs))) break;
            if (!(ok = mbar_wait(full_a(s), rg.ph, s_abort, kMmaSleepNs))) break;
            tc_fence_after();
            const uint32_t a0 = stage0 + s * p.stage_bytes;
            const uint32_t b0 = a0 + p.a_bytes;
#pragma unroll
            for (int a = 0; a < kAtoms; ++a) {
#pragma unroll
              for (int ks = 0; ks < kAtomK / 16; ++ks) {
                const uint64_t bdesc = sdesc_sw128(b0 + a * p.x_atom_bytes + ks * 32);
#pragma unroll
                for (int h = 0; h < MH; ++h) {
                  umma_bf16(dcol + (ii * MH + h) * p.nt,
                            sdesc_sw128(a0 + (a * MH + h) * kHalfBytes + ks * 32), bdesc, p.idesc,
                            (kc | a | ks) != 0);
                }
              }
            }
            umma_commit(empty(s));
          }
        }
        if (ok) umma_commit(tmem_full(b));
      }
      // All issued MMAs have completed once this commit arrives.
      umma_commit(drain);
      const uint64_t t0 = global_ns();
      while (!mbar_try_wait(drain, 0) && global_ns() - t0 < p.timeout_ns) {
      }
    }
  } else if (warp < kFirstHashWarp) {
    // ---------------------------------------------------------------- epilogue
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    Ring tb;
    for (int64_t u = blockIdx.x; u < p.units; u += gridDim.x, tb.next(p.nbuf)) {
      const Unit un = decode(p, u, MH);
      const int b = tb.s;
      // One thread polls (backing off longer when TMEM is double-buffered and the
      // epilogue is off the critical path); the other 127 epilogue threads block
      // on a named barrier, which takes no issue slots.
      if (threadIdx.x == kEpilogueFirstThread)
        mbar_wait(tmem_full(b), tb.ph, s_abort, p.nbuf == 2 ? 2000 : 300);
      named_barrier_sync(kEpilogueBarrier, kEpilogueThreads);
      __syncwarp();
      if (s_abort->abort) break;
      tc_fence_after();
      const uint32_t dcol = tmem + b * cols_per_buf + (static_cast<uint32_t>(quarter * 32) << 16);
      for (int ii = 0; ii < (kG1 ? 1 : un.gcount); ++ii) {
        const int64_t i = un.i0 + ii;
        const uint64_t seed = static_cast<uint64_t>(__ldg(p.seeds + i));
#pragma unroll
        for (int h = 0; h < MH; ++h) {
          const int64_t j = un.m0 + h * 128 + row;
          const bool jok = j < p.out;
          float bias = 0.f;
          if (jok && p.b != nullptr) {
            const float bj = p.b_bf16
                                 ? __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(p.b)[j])
                                 : reinterpret_cast<const float*>(p.b)[j];
            const uint64_t bidx =
                p.offset + static_cast<uint64_t>(p.out) * static_cast<uint64_t>(p.in) +
                static_cast<uint64_t>(j);
            bias = fmaf(p.sigma, noise_at_kind<kKind>(seed, bidx), bj);
          }
          // Y[i, n, j] for the unit's batch rows n = n0 + c0 + q: one row pointer
          // per 16 columns, batch rows `out` elements apart.
          using YT = typename std::conditional<kYBf16, unsigned short, float>::type;
          YT* yrow = reinterpret_cast<YT*>(p.y) + (i * p.batch + un.n0) * p.out + j;
          const int64_t ystride = p.out;
          const int n_left = static_cast<int>(min(static_cast<int64_t>(p.nt), p.batch - un.n0));
          const bool tanh_act = p.act == VN_ACT_TANH;
          for (int c0 = 0; c0 < p.nt; c0 += 16, yrow += 16 * ystride) {
            uint32_t v[16];
            tmem_ld16(dcol + (ii * MH + h) * p.nt + c0, v);
            tmem_wait_ld();
            if (jok) {
              const int valid = n_left - c0;  // columns of this group that are batch rows
              // The epilogue warps share the schedulers with the hashing warps, so the
              // common case (all 16 columns are batch rows, no activation) is one
              // straight run of adds, conversions and stores; the activation and the
              // ragged last group take the general loop.
              if (valid >= 16 && !tanh_act) {
#pragma unroll
                for (int q = 0; q < 16; ++q) store_y<kYBf16>(yrow + q * ystride, __uint_as_float(v[q]) + bias);
              } else {
#pragma unroll
                for (int q = 0; q < 16; ++q) {
                  if (q < valid) {
                    float val = __uint_as_float(v[q]) + bias;
                    if (tanh_act) val = tanhf(val);
                    store_y<kYBf16>(yrow + q * ystride, val);
                  }
                }
              }
            }
          }
        }
      }
      tc_fence_before();
      mbar_arrive(tmem_empty(b));
    }
  } else {
    // ----------------------------------------------------------------- hashing
    // Thread t writes 16-byte chunk (t & 7) of rows (t >> 3) + kRowsPerPass*q of
    // each atom of the (128*MH)-row A tile, q < kCPT: one 128-byte row per 8 lanes,
    // so each quarter-warp store covers all 32 banks once (the swizzle permutes the
    // chunks within a row). The two 128-row halves of an MH=2 atom are contiguous,
    // so row r sits at (r >> 3)*1024 + (r & 7)*128 for any r < 256; atom a of the
    // stage starts a*MH*16 KB in. A thread makes kCPT*kAtoms chunks of 8 elements
    // per stage.
    constexpr int kRowsPerPass = kHashThreads / 8;          // rows covered by one chunk round
    constexpr int kCPT = MH * 128 / kRowsPerPass;           // row passes per atom
    using Raw = typename std::conditional<kWBf16, RawBf16, RawF32>::type;
    const int t = threadIdx.x - kFirstHashWarp * 32;
    const int cc = t & 7;
    const int r8 = (t >> 3) & 7;
    const uint32_t soff0 = static_cast<uint32_t>(t >> 6) * 1024u + r8 * 128u + ((cc ^ r8) << 4);
    const int row0 = t >> 3;
    auto soff = [&](int q, int a) {
      return soff0 + q * (kRowsPerPass * 128u) + static_cast<uint32_t>(a * MH) * kHalfBytes;
    };
    auto rowq = [&](int q) { return row0 + q * kRowsPerPass; };
    const float sigma = p.sigma;
    // Uniform kind: W + sigma*n = fma(sigma, 1 + u, W - 1.5*sigma). Gaussian kind:
    // W + sigma*G = fma(sigma * kGaussScale, unit, W), unit from the finalizer's halves.
    const float shift = kKind == kGaussian ? 0.f : -1.5f * sigma;
    const float sigma_unit = kKind == kGaussian ? sigma * kGaussScale : sigma;
    const uint32_t g_lo = p.g_lo, g_hi = p.g_hi, one = p.one;

    // This thread's chunk (q, a) inside a staged W tile (rows of kKC k: 128*kAtoms
    // bytes in bf16, 256*kAtoms in fp32). In fp32 the two 16-byte halves are read in
    // an order that depends on cc, so the 8 threads of a row hit distinct banks.
    constexpr uint32_t kWElem = kWBf16 ? 2u : 4u;
    constexpr uint32_t kWRow = kKC * kWElem;
    const uint32_t wfirst = kWBf16 ? 0u : ((cc >> 2) & 1u) * 16u;
    auto woff = [&](int q, int a) {
      return static_cast<uint32_t>(rowq(q)) * kWRow + (a * kAtomK + cc * 8) * kWElem;
    };
    auto load_w = [&](uint32_t addr, Raw& r) {
      if constexpr (kWBf16) {
        r.a = ld_shared_v4(addr);
      } else {
        const uint4 h0 = ld_shared_v4(addr + wfirst);
        const uint4 h1 = ld_shared_v4(addr + (wfirst ^ 16u));
        const uint4 lo = wfirst ? h1 : h0;
        const uint4 hi = wfirst ? h0 : h1;
        r.a = make_float4(__uint_as_float(lo.x), __uint_as_float(lo.y), __uint_as_float(lo.z),
                          __uint_as_float(lo.w));
        r.b = make_float4(__uint_as_float(hi.x), __uint_as_float(hi.y), __uint_as_float(hi.z),
                          __uint_as_float(hi.w));
      }
    };
    // State term step from one k chunk to the next: kKC * GAMMA mod 2^64.
    constexpr uint64_t kChunkStep = static_cast<uint64_t>(kKC) * kGamma;
    // From a chunk's last element (k + 7) to the next k chunk's first (k + kKC).
    constexpr uint64_t kChunkHop = static_cast<uint64_t>(kKC - 7) * kGamma;

    // Ring positions (slot, parity) of the stages and of the W tiles; barrier
    // addresses are formed from them directly.
    const uint32_t S32 = static_cast<uint32_t>(S);
    const uint32_t stage_bytes = p.stage_bytes;
    const uint32_t fa0 = full_a(0), em0 = empty(0), fw0 = full_w(0), ew0 = empty_w(0);
    const uint32_t a_this = stage0 + soff(0, 0);   // this thread's first chunk in stage 0
    const uint32_t w_this = wslot0 + woff(0, 0);
    const uint32_t w_bytes = p.w_bytes;
    const uint32_t w_slots = static_cast<uint32_t>(p.w_slots);
    const int k_chunks = p.k_chunks;
    uint32_t s = 0, ph = 0, ws = 0, wph = 0;
    // Test hook: the stage at which this thread skips its arrive (-1: never).
    int withhold_at = (kHook && p.withhold_stage >= 0 && p.withhold_stage < 0x7FFFFFFF &&
                       blockIdx.x == 0 && t == 0) ? static_cast<int>(p.withhold_stage) : -1;
    for (int64_t u = blockIdx.x; u < p.units; u += gridDim.x) {
      const Unit un = decode(p, u, MH);
      const int64_t* seedp = p.seeds + un.i0;
      // (offset + j*in + k + 1) * GAMMA of each chunk's first element, k chunk 0;
      // advanced by kChunkStep per k chunk. With one individual per unit its seed
      // is added here once, and the halves blo:bhi carry each chunk's state chain
      // from one k chunk to the next.
      uint64_t bst[kCPT][kAtoms];
      uint32_t blo[kCPT][kAtoms], bhi[kCPT][kAtoms];
      const uint64_t seed0 = kG1 ? static_cast<uint64_t>(__ldg(seedp)) : 0ull;
#pragma unroll
      for (int q = 0; q < kCPT; ++q) {
#pragma unroll
        for (int a = 0; a < kAtoms; ++a) {
          bst[q][a] = seed0 + index_term(p.offset +
                                         static_cast<uint64_t>(un.m0 + rowq(q)) *
                                             static_cast<uint64_t>(p.in) +
                                         static_cast<uint64_t>(a * kAtomK + cc * 8));
          blo[q][a] = static_cast<uint32_t>(bst[q][a]);
          bhi[q][a] = static_cast<uint32_t>(bst[q][a] >> 32);
        }
      }
      // This thread's chunks of a staged W tile (wb: its first one). fp32 W is
      // kept as W - 1.5*sigma and perturbed with one FMA per element; bf16 W
      // stays packed and each element is formed as fp32(bf16 W) + sigma*n with
      // one mixed-precision add (no unpacking on the integer pipe). Chunks
      // outside the matrix (row >= out or k >= in, only at ragged edges) are
      // TMA's zero fill, so their values are finite: their X columns are zero
      // fill too (k >= in) or their output rows are never stored (row >= out),
      // and no masking is needed below.
      auto load_stage_w = [&](uint32_t wb, Raw (&wraw)[kCPT][kAtoms], float (&wm)[kCPT][kAtoms][8]) {
#pragma unroll
        for (int q = 0; q < kCPT; ++q) {
#pragma unroll
          for (int a = 0; a < kAtoms; ++a) {
            load_w(wb + woff(q, a) - woff(0, 0), wraw[q][a]);
            if constexpr (!kWBf16) unpack_shift(wraw[q][a], shift, wm[q][a]);
          }
        }
      };
      // One stage of one individual: W'_i of this thread's chunks, packed to
      // bf16 and stored to the A tile whose chunk for this thread is at a0.
      auto hash_stage = [&](uint32_t a0, uint64_t seed, const Raw (&wraw)[kCPT][kAtoms],
                            const float (&wm)[kCPT][kAtoms][8]) {
#pragma unroll
        for (int q = 0; q < kCPT; ++q) {
#pragma unroll
          for (int a = 0; a < kAtoms; ++a) {
            // One individual per unit: the chunk's state chain runs in place in
            // blo:bhi, and the step after its last element adds (kKC - 7) * GAMMA,
            // which lands on the next k chunk's first. Otherwise each individual
            // starts from bst + seed.
            uint32_t slo, shi;
            if constexpr (kG1) {
              slo = blo[q][a];
              shi = bhi[q][a];
            } else {
              const uint64_t st0 = bst[q][a] + seed;
              slo = static_cast<uint32_t>(st0);
              shi = static_cast<uint32_t>(st0 >> 32);
            }
            float pv[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              // The element's noise term: the uniform kind as 1 + u (its -1.5 rides on
              // the shift), the Gaussian kind as the unit Box-Muller value.
              float unit;
              if constexpr (kKind == kGaussian) {
                uint32_t zlo, zhi;
                mix64_halves(slo, shi, zlo, zhi);
                unit = gaussian_unit(zlo, zhi);
              } else {
                unit = __uint_as_float(mix_to_one_plus_u(slo, shi));
              }
              if constexpr (kWBf16) {
                // sigma*n = fma(sigma, 1 + u, -1.5*sigma), then + W straight from its bf16 bits.
                const float tt = fmaf(sigma_unit, unit, shift);
                const uint32_t wv = (e & 4) ? ((e & 2) ? wraw[q][a].a.w : wraw[q][a].a.z)
                                            : ((e & 2) ? wraw[q][a].a.y : wraw[q][a].a.x);
                pv[e] = (e & 1) ? add_bf16_f32<true>(wv, tt) : add_bf16_f32<false>(wv, tt);
              } else {
                pv[e] = fmaf(sigma_unit, unit, wm[q][a][e]);
              }
              if (e < 7)
                add64_madc(slo, shi, g_lo, g_hi, one);
              else if constexpr (kG1)
                add64_madc(slo, shi, static_cast<uint32_t>(kChunkHop),
                           static_cast<uint32_t>(kChunkHop >> 32), one);
            }
            if constexpr (kG1) {
              blo[q][a] = slo;
              bhi[q][a] = shi;
            }
            st_shared_v4(a0 + soff(q, a) - soff(0, 0), pack_bf16x2(pv[0], pv[1]),
                         pack_bf16x2(pv[2], pv[3]), pack_bf16x2(pv[4], pv[5]),
                         pack_bf16x2(pv[6], pv[7]));
          }
        }
      };

      if constexpr (kFix) {
        // Two stages, one W tile, an even number of k chunks per unit: every
        // unit starts on stage 0 with W parity 0, so within a pair of k chunks
        // the stage slot and the W parity are both h, and only the stage
        // parity (flipped once per pair) is carried.
        for (int kc = 0; kc < k_chunks; kc += 2) {
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            if (!mbar_wait(fw0, static_cast<uint32_t>(h), s_abort)) goto hashing_done;
            float wm[kCPT][kAtoms][8];
            Raw wraw[kCPT][kAtoms];
            load_stage_w(w_this, wraw, wm);
            // The W tile is rewritten by TMA (the async proxy): order this
            // thread's generic-proxy reads of it before that write.
            fence_proxy_async_smem();
            mbar_arrive(ew0);
            if (!mbar_wait(em0 + 8u * h, ph ^ 1u, s_abort)) goto hashing_done;
            hash_stage(h ? a_this + stage_bytes : a_this, 0ull, wraw, wm);
            fence_proxy_async_smem();
            mbar_arrive(fa0 + 8u * h);
          }
          ph ^= 1u;
        }
      } else {
        for (int kc = 0; kc < k_chunks; ++kc) {
          // This stage group's W chunks, shared by its G individuals.
          if (!mbar_wait(fw0 + 8u * ws, wph, s_abort)) goto hashing_done;
          float wm[kCPT][kAtoms][8];
          Raw wraw[kCPT][kAtoms];
          load_stage_w(w_this + ws * w_bytes, wraw, wm);
          // The slot's next tile is written by TMA (the async proxy): order this
          // thread's generic-proxy reads of it before that write. Without the
          // fence a late warp's reads could return the next tile's values.
          fence_proxy_async_smem();
          mbar_arrive(ew0 + 8u * ws);
          if (++ws == w_slots) { ws = 0; wph ^= 1u; }
          for (int ii = 0; ii < (kG1 ? 1 : un.gcount); ++ii) {
            const uint64_t seed = kG1 ? 0ull : static_cast<uint64_t>(__ldg(seedp + ii));
            if (!mbar_wait(em0 + 8u * s, ph ^ 1u, s_abort)) goto hashing_done;
            hash_stage(a_this + s * stage_bytes, seed, wraw, wm);
            fence_proxy_async_smem();
            if constexpr (kHook) {
              if (withhold_at != 0) mbar_arrive(fa0 + 8u * s);
              if (withhold_at >= 0) --withhold_at;
            } else {
              mbar_arrive(fa0 + 8u * s);
            }
            if (++s == S32) { s = 0; ph ^= 1u; }
          }
          if constexpr (!kG1) {
#pragma unroll
            for (int q = 0; q < kCPT; ++q) {
#pragma unroll
              for (int a = 0; a < kAtoms; ++a) bst[q][a] += kChunkStep;
            }
          }
        }
      }
    }
  hashing_done:;
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ---------------------------------------------------------------- host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

template <int MH, bool kW, bool kY, bool kHook, int kKind, bool kG1, int kAtoms, bool kFix = false>
cudaError_t launch_kernel(const CUtensorMap& xmap, const CUtensorMap& wmap, const TcParams& p,
                          int grid, size_t smem, cudaStream_t stream) {
  auto fn = linear_tc_kernel<MH, kW, kY, kHook, kKind, kG1, kAtoms, kFix>;
  static SmemRecord configured;
  const cudaError_t err = ensure_dynamic_smem(reinterpret_cast<const void*>(fn), smem, configured);
  if (err != cudaSuccess) return err;
  fn<<<grid, kThreads, smem, stream>>>(xmap, wmap, p);
  return cudaGetLastError();
}

// One individual per unit (the whole TMEM buffer for one batch tile): the
// individual loops of every role have a single, compile-time iteration. `atoms`:
// 64-k swizzle atoms per stage (1 or 2).
template <int MH, bool kW, bool kY, bool kHook, int kKind = kUniform>
cudaError_t launch_typed(const CUtensorMap& xmap, const CUtensorMap& wmap, const TcParams& p,
                         int atoms, int grid, size_t smem, cudaStream_t stream) {
  if (atoms == 2) {
    // The fixed loop for the uniform kind only: the Gaussian kind's longer chunk
    // body runs slower in it (5.75 against 5.51 ms on 256 x 256 x 4096^2).
    if constexpr (kW && !kHook && kKind == kUniform) {
      if (p.g == 1 && p.stages == 2 && p.w_slots == 1 && p.k_chunks % 2 == 0)
        return launch_kernel<MH, kW, kY, kHook, kKind, true, 2, true>(xmap, wmap, p, grid, smem, stream);
    }
    if (p.g == 1 && !kHook)
      return launch_kernel<MH, kW, kY, kHook, kKind, true, 2>(xmap, wmap, p, grid, smem, stream);
    return launch_kernel<MH, kW, kY, kHook, kKind, false, 2>(xmap, wmap, p, grid, smem, stream);
  }
  if (p.g == 1 && !kHook)
    return launch_kernel<MH, kW, kY, kHook, kKind, true, 1>(xmap, wmap, p, grid, smem, stream);
  return launch_kernel<MH, kW, kY, kHook, kKind, false, 1>(xmap, wmap, p, grid, smem, stream);
}

}  // namespace

bool linear_tc_applies(const void* x, vn_dtype x_dt, const void* w, vn_dtype w_dt, int64_t batch,
                       int64_t in, int64_t out) {
  (void)w_dt;
  const int64_t kMaxCoord = (int64_t{1} << 31) - 1;
  return x_dt == VN_BF16 && batch >= 1 && batch <= kMaxCoord && in >= 8 && in % 8 == 0 &&
         in <= kMaxCoord && out >= 1 && out <= kMaxCoord && reinterpret_cast<uintptr_t>(x) % 16 == 0 &&
         reinterpret_cast<uintptr_t>(w) % 16 == 0;
}

cudaError_t launch_linear_tc(const LinearArgs& a, cudaStream_t stream) {
  return launch_linear_tc_hook(a, stream, -1, kTimeoutNs);
}

cudaError_t launch_linear_tc_hook(const LinearArgs& a, cudaStream_t stream, long long withhold_stage,
                                  unsigned long long timeout_ns) {
  DeviceInfo dev;
  cudaError_t err = device_info(&dev);
  if (err != cudaSuccess) return err;
  if (a.pop > (int64_t{1} << 31) - 1) return cudaErrorInvalidValue;
  PFN_cuTensorMapEncodeTiled_v12000 encode = encode_fn();
  if (encode == nullptr) return cudaErrorNotSupported;

  TcParams p;
  std::memset(&p, 0, sizeof(p));
  const int64_t nt = std::min<int64_t>(256, (a.batch + 15) / 16 * 16);
  const bool wbf = a.w_dt == VN_BF16;
  // 128-row units: each unit's accumulators fit in 256 TMEM columns, so TMEM is
  // double-buffered and the epilogue of one unit overlaps the next unit's MMAs.
  // (256-row units halve the X traffic per element but then fill all 512
  // columns; measured slower on the 256-batch workload.)
  const int mh = 1;
  int g = static_cast<int>(std::max<int64_t>(1, 256 / (mh * nt)));
  g = static_cast<int>(std::min<int64_t>(g, a.pop));
  p.b = a.b; p.seeds = a.seeds; p.y = a.y;
  p.pop = a.pop; p.batch = a.batch; p.in = a.in; p.out = a.out;
  p.offset = a.offset; p.sigma = a.sigma;
  p.b_bf16 = (a.b != nullptr && a.b_dt == VN_BF16) ? 1 : 0;
  p.act = a.act;
  p.nt = static_cast<int>(nt);
  p.g = g;
  p.nbuf = (static_cast<int64_t>(g) * mh * nt <= kTmemCols / 2) ? 2 : 1;
  // alignment slack + barriers (at most 8 stages) + TMEM address + wait control
  const size_t fixed = 1024 + 8 * (3 * 8 + 9) + 8 + 16;
  // Stage shape: two 64-k atoms per stage (32 elements per hashing thread per
  // stage) with a ring of two W tiles, else with one W tile, else one atom per
  // stage with two W tiles -- the first that leaves room for two stages.
  const uint32_t welem = wbf ? 2u : 4u;
  int atoms = 0, w_slots = 0, stages = 0;
  static const int kPlans[3][2] = {{2, 2}, {2, 1}, {1, 2}};  // {atoms, W slots}
  for (const auto& c : kPlans) {
    const int64_t stage = static_cast<int64_t>(c[0]) * (static_cast<int64_t>(mh) * kHalfBytes + nt * 128);
    const int64_t wtile = 128 * static_cast<int64_t>(kAtomK) * c[0] * welem;
    const int64_t st = std::min<int64_t>(
        8, (static_cast<int64_t>(dev.smem_optin) - static_cast<int64_t>(fixed) - c[1] * wtile) / stage);
    if (st >= 2) {
      atoms = c[0];
      w_slots = c[1];
      stages = static_cast<int>(st);
      break;
    }
  }
  if (stages < 2) return cudaErrorInvalidConfiguration;
  const int kc_len = kAtomK * atoms;
  p.x_atom_bytes = static_cast<uint32_t>(nt) * 128u;
  p.a_bytes = static_cast<uint32_t>(atoms * mh) * kHalfBytes;
  p.stage_bytes = p.a_bytes + static_cast<uint32_t>(atoms) * p.x_atom_bytes;
  p.w_bytes = 128u * static_cast<uint32_t>(kc_len) * welem;
  p.w_slots = w_slots;
  p.stages = stages;
  p.k_chunks = static_cast<int>((a.in + kc_len - 1) / kc_len);
  p.m_tiles = (a.out + 128 * mh - 1) / (128 * mh);
  p.n_tiles = (a.batch + nt - 1) / nt;
  const int64_t groups = (a.pop + g - 1) / g;
  p.units = groups * p.n_tiles * p.m_tiles;
  p.units32 = (p.units + dev.sm_count) <= 0xFFFFFFFFll ? 1 : 0;
  p.x_shared = a.x_shared;
  p.timeout_ns = timeout_ns;
  p.g_lo = kGammaLo;
  p.g_hi = kGammaHi;
  p.one = 1u;
  p.withhold_stage = withhold_stage;
  // Instruction descriptor: fp32 accumulator, bf16 A and B, both K-major,
  // N = nt (bits 17-22, N >> 3), M = 128 (bits 24-28, M >> 4).
  p.idesc = (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(nt >> 3) << 17) |
            (static_cast<uint32_t>(128 >> 4) << 24);

  // X as a 3-D tensor [pop or 1][batch][in] of bf16; box = 64 k (one swizzle atom)
  // x nt rows x 1.
  CUtensorMap xmap;
  std::memset(&xmap, 0, sizeof(xmap));
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(a.in), static_cast<cuuint64_t>(a.batch),
                              static_cast<cuuint64_t>(a.x_shared ? 1 : a.pop)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(a.in) * 2,
                                 static_cast<cuuint64_t>(a.in) * 2 * static_cast<cuuint64_t>(a.batch)};
  const cuuint32_t box[3] = {static_cast<cuuint32_t>(kAtomK), static_cast<cuuint32_t>(nt), 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult cr = encode(&xmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(a.x),
                             dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (cr != CUDA_SUCCESS) return cudaErrorInvalidValue;

  // W as a 2-D tensor [out][in] of its dtype; box = 64 * atoms k x 128 rows, no
  // swizzle (the hashing warps read it with plain shared loads). Rows >= out
  // and k >= in arrive as zeros.
  CUtensorMap wmap;
  std::memset(&wmap, 0, sizeof(wmap));
  const cuuint64_t wdims[2] = {static_cast<cuuint64_t>(a.in), static_cast<cuuint64_t>(a.out)};
  const cuuint64_t wstrides[1] = {static_cast<cuuint64_t>(a.in) * (wbf ? 2 : 4)};
  const cuuint32_t wbox[2] = {static_cast<cuuint32_t>(kc_len), 128};
  const cuuint32_t westr[2] = {1, 1};
  const CUresult wr = encode(&wmap,
                             wbf ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                             2, const_cast<void*>(a.w), wdims, wstrides, wbox, westr,
                             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (wr != CUDA_SUCCESS) return cudaErrorInvalidValue;

  const size_t smem = fixed + static_cast<size_t>(stages) * p.stage_bytes +
                      static_cast<size_t>(w_slots) * p.w_bytes;
  const int grid = static_cast<int>(std::min<int64_t>(p.units, dev.sm_count));
  const bool ybf = a.y_dt == VN_BF16;
  if (withhold_stage >= 0) {
    // The test hook has one instance: bf16 W and Y.
    if (!(wbf && ybf)) return cudaErrorInvalidValue;
    return launch_typed<1, true, true, true>(xmap, wmap, p, atoms, grid, smem, stream);
  }
  if (a.kind == kGaussian) {
    if (wbf) {
      return ybf ? launch_typed<1, true, true, false, kGaussian>(xmap, wmap, p, atoms, grid, smem, stream)
                 : launch_typed<1, true, false, false, kGaussian>(xmap, wmap, p, atoms, grid, smem, stream);
    }
    return launch_typed<1, false, false, false, kGaussian>(xmap, wmap, p, atoms, grid, smem, stream);
  }
  if (wbf) {
    return ybf ? launch_typed<1, true, true, false>(xmap, wmap, p, atoms, grid, smem, stream)
               : launch_typed<1, true, false, false>(xmap, wmap, p, atoms, grid, smem, stream);
  }
  return launch_typed<1, false, false, false>(xmap, wmap, p, atoms, grid, smem, stream);
}

cudaError_t take_device_status(unsigned int* status, cudaStream_t stream) {
  cudaError_t err = cudaMemcpyFromSymbolAsync(status, g_device_status, sizeof(unsigned int), 0,
                                              cudaMemcpyDeviceToHost, stream);
  if (err != cudaSuccess) return err;
  err = cudaStreamSynchronize(stream);
  if (err != cudaSuccess) return err;
  if (*status != 0) {
    const unsigned int zero = 0;
    err = cudaMemcpyToSymbolAsync(g_device_status, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice,
                                  stream);
    if (err == cudaSuccess) err = cudaStreamSynchronize(stream);
  }
  return err;
}

}  // namespace vn
