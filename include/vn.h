/*
 * vn.h -- C ABI of the virtual-noise evolution-strategies library (libvn.so).
 *
 * The library computes, on one CUDA device, the population evolution-strategies
 * step with virtual (never materialised) weight noise described on the EvoX API
 * page "evox.triton_kernels.kernels.virtual_noise":
 *
 *   forward   Y[i] = X[i] @ (W + sigma*N_i)^T + (b + sigma*nb_i)      (module description)
 *   gradient  grad_W[j,k] = sum_i f_i * N_i[j,k] / (pop*sigma)        (module description)
 *   noise     N_i[j,k] = PRNG(seed_i, offset + j*in + k),             ("Noise indexing scheme")
 *             nb_i[j]  = PRNG(seed_i, offset + out*in + j)
 *
 * PRNG(seed, idx) -- the definition every entry point follows, bit for bit:
 *   GAMMA = 0x9E3779B97F4A7C15 (11400714819323198485, "_SPLITMIX64_GAMMA");
 *   z = seed + (idx + 1) * GAMMA                         (mod 2^64)
 *   z = (z ^ (z >> 30)) * GAMMA; z = (z ^ (z >> 27)) * GAMMA; z ^= z >> 31
 *       (logical shifts, products mod 2^64; "_splitmix64_step" as printed)
 *   PRNG = (lo32(z) >> 9) * 2^-23 - 0.5,  a float32 value in [-0.5, 0.5)
 *       (low 32 bits of the hash, "_cpu_normal_noise"; the top 23 of them, so
 *        the value is exact in float32 and never reaches 0.5).
 * The state formula (the idx-th output of a splitmix64 generator seeded with
 * seed) is this library's reading: the page does not say how seed and index
 * are combined. Seeds are signed 64-bit integers taken mod 2^64. The element
 * index offset + j*in + k is evaluated in unsigned 64-bit arithmetic and wraps.
 *
 * Conventions shared by every entry point
 *   - Every tensor pointer is a CUDA device pointer owned by the caller, to a
 *     dense row-major array on the current device. Nothing is copied, retained
 *     or freed. fp32 arrays must be 4-byte aligned, bf16 arrays 2-byte aligned,
 *     seeds 8-byte aligned (else VN_ERR_ALIGN).
 *   - All work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *     stream) and is asynchronous: a VN_OK return means the arguments were
 *     valid and the kernel was launched, not that it has finished.
 *   - Arguments are validated on the host before anything is launched. A call
 *     that fails validation returns its status and launches nothing.
 *   - An output array may not share memory with an input array of the same
 *     call, nor with another output: a call whose arrays overlap that way
 *     returns VN_ERR_VALUE and launches nothing.
 *   - A size of 0 in an output dimension is valid and launches nothing (the
 *     pointers of empty arrays may then be NULL).
 *   - Kernels that wait on on-chip barriers bound every wait. A wait that runs
 *     out records VN_ERR_TIMEOUT in a device-side status word, which
 *     vn_device_status() reports; the kernel returns without hanging the GPU.
 *   - The library allocates no device memory at call time.
 */
#ifndef VN_H
#define VN_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum vn_status {
  VN_OK = 0,
  VN_ERR_NULL = 1,     /* a required pointer is NULL                                */
  VN_ERR_SHAPE = 2,    /* a size is negative, or pop < 1 where an estimate needs it   */
  VN_ERR_DTYPE = 3,    /* unsupported dtype or dtype combination                    */
  VN_ERR_VALUE = 4,    /* sigma not finite, sigma == 0 for a gradient, an unknown    */
                       /* enum, or an output overlapping an input of the call       */
  VN_ERR_ALIGN = 5,    /* a pointer is not aligned to its element size              */
  VN_ERR_OVERFLOW = 6, /* a size product does not fit in int64                      */
  VN_ERR_TIMEOUT = 7,  /* a device-side bounded wait ran out (vn_device_status)     */
  VN_ERR_CUDA = 8,     /* a CUDA runtime call failed (vn_last_error_message)        */
  VN_ERR_DEVICE = 9,   /* the requested path needs a compute-capability 10.x GPU    */
  VN_ERR_PATH = 10     /* the forced forward path cannot run these arguments        */
} vn_status;

typedef enum vn_dtype { VN_F32 = 0, VN_BF16 = 1 } vn_dtype;

/* Forward kernel selection for vn_perturbed_linear_ex. */
typedef enum vn_path {
  VN_PATH_AUTO = 0,  /* VN_PATH_TC when it applies and batch >= 16, else FFMA      */
  VN_PATH_FFMA = 1,  /* CUDA-core path: any dtypes, any batch                       */
  VN_PATH_TC = 2     /* tcgen05/TMEM path: x bf16, in % 8 == 0, x and w 16-byte     */
                     /* aligned, pop, batch, in and out below 2^31                 */
} vn_path;

/* Noise distribution of the _ex dump and gradient entry points. */
typedef enum vn_noise {
  VN_NOISE_UNIFORM = 0,  /* PRNG(seed, idx) above: the page's centered uniform, bit-exact  */
  VN_NOISE_GAUSSIAN = 1  /* Box-Muller on the same finalizer output z (a variant; the page  */
                         /* names Gaussian noise as the costly alternative):                */
                         /*   u1 = 1 - (hi32(z) >> 9) 2^-23,  u2 = (lo32(z) >> 9) 2^-23,     */
                         /*   G = sqrt(-2 ln u1) cos(2 pi u2)                                */
                         /* computed with the hardware log2 and cos: |error| <= 6e-4 where   */
                         /* u1 is within 2^-12 of 1 (G near 0), about 1e-6 elsewhere.        */
} vn_noise;

/* Element-wise activation applied to Y after the bias (vn_perturbed_linear_ex). */
typedef enum vn_act { VN_ACT_NONE = 0, VN_ACT_TANH = 1 } vn_act;

/*
 * vn_perturbed_linear -- "virtual_perturbed_linear" (API entry of the page):
 *     Y[i, r, :] = X[i, r, :] @ (W + sigma*N_i)^T + (b + sigma*nb_i)
 * x       [pop, batch, in] of x_dt, or [batch, in] when x_shared != 0 (the same
 *         input for every individual).
 * w       [out, in] of w_dt.                 b  [out] of b_dt, or NULL: then
 *         there is no bias term and no bias noise.
 * seeds   [pop] int64.                       y  [pop, batch, out] of y_dt.
 * offset  flat element offset of this weight block (compute_offsets); the bias
 *         noise is read at offset + out*in + j.
 * dtypes  x, w, b: VN_F32 or VN_BF16. y_dt must be VN_BF16 when x and w are
 *         both bf16 and VN_F32 otherwise (torch's result type of x and w).
 * Arithmetic: W + sigma*N_i is formed in fp32 per element. On the tensor-core
 * path it is rounded to bf16 and contracted with bf16 x, accumulating in fp32;
 * on the FFMA path everything is fp32. in == 0 gives Y = b + sigma*nb_i.
 */
vn_status vn_perturbed_linear(const void* x, vn_dtype x_dt, int x_shared,
                              const void* w, vn_dtype w_dt,
                              const void* b, vn_dtype b_dt,
                              const int64_t* seeds, int64_t pop, int64_t batch,
                              int64_t in, int64_t out, double sigma, uint64_t offset,
                              void* y, vn_dtype y_dt, void* stream);

/* vn_perturbed_linear with an explicit kernel choice and a fused activation
 * (applied after the bias). VN_PATH_TC returns VN_ERR_PATH when its conditions
 * do not hold and VN_ERR_DEVICE on a device that is not compute capability 10.x.
 * On the CUDA-core path, VN_PATH_AUTO with fp32 W and b, batch <= 8 and at least
 * as many individuals as the device has SMs runs the kernel of vn_perturbed_mlp
 * with one layer (its individuals share every W chunk they load); VN_PATH_FFMA
 * always runs the single-layer kernel. Both compute in fp32. */
vn_status vn_perturbed_linear_ex(const void* x, vn_dtype x_dt, int x_shared,
                                 const void* w, vn_dtype w_dt,
                                 const void* b, vn_dtype b_dt,
                                 const int64_t* seeds, int64_t pop, int64_t batch,
                                 int64_t in, int64_t out, double sigma, uint64_t offset,
                                 void* y, vn_dtype y_dt, vn_path path, vn_act act,
                                 void* stream);

/*
 * vn_perturbed_linear_kind -- vn_perturbed_linear_ex with a choice of noise
 * distribution: N_i and nb_i are noise_kind(seed_i, index) at the same indices
 * (VN_NOISE_UNIFORM: vn_perturbed_linear_ex exactly). VN_NOISE_GAUSSIAN (the
 * Box-Muller variant of vn_noise, within its stated error) runs on the
 * tensor-core kernel (VN_PATH_TC, or VN_PATH_AUTO with its conditions and batch
 * >= 16) or on the chain kernel of vn_perturbed_mlp with one layer (fp32 W and b,
 * batch <= 8, a layer that fits its shared memory; VN_PATH_AUTO or VN_PATH_FFMA);
 * other Gaussian calls return VN_ERR_PATH. An unknown kind returns VN_ERR_VALUE.
 */
vn_status vn_perturbed_linear_kind(const void* x, vn_dtype x_dt, int x_shared,
                                   const void* w, vn_dtype w_dt,
                                   const void* b, vn_dtype b_dt,
                                   const int64_t* seeds, int64_t pop, int64_t batch,
                                   int64_t in, int64_t out, double sigma, uint64_t offset,
                                   void* y, vn_dtype y_dt, vn_path path, vn_act act,
                                   vn_noise kind, void* stream);

/*
 * vn_weight_gradient -- "virtual_weight_gradient" (API entry of the page):
 *     grad_w[j, k] = sum_i fitness[i] * N_i[j, k] / (pop * sigma)
 * fitness [pop] fp32, seeds [pop] int64, grad_w [out, in] fp32 (written, not
 * accumulated into). N_i[j,k] is read at offset + j*in + k, the same elements
 * vn_perturbed_linear perturbs. pop >= 1; sigma finite and nonzero. The sum
 * over individuals is accumulated in fp32 in a fixed order (deterministic) and
 * multiplied by fp32(1 / (pop*sigma)).
 */
vn_status vn_weight_gradient(const float* fitness, const int64_t* seeds, int64_t pop,
                             int64_t out, int64_t in, double sigma, uint64_t offset,
                             float* grad_w, void* stream);

/*
 * vn_bias_gradient -- "virtual_bias_gradient" (API entry of the page):
 *     grad_b[j] = sum_i fitness[i] * nb_i[j] / (pop * sigma),  nb_i[j] at offset + j.
 * `offset` already points at the bias region: pass weight_offset + out*in to
 * match the bias noise of vn_perturbed_linear. Same conventions as
 * vn_weight_gradient.
 */
vn_status vn_bias_gradient(const float* fitness, const int64_t* seeds, int64_t pop,
                           int64_t out, double sigma, uint64_t offset,
                           float* grad_b, void* stream);

/*
 * vn_noise_dump -- the "_cpu_normal_noise" contract (API entry of the page):
 *     out[i, t] = PRNG(seed_i, offset + t),  out [pop, n] fp32.
 * Bit-exact with the definition above.
 */
vn_status vn_noise_dump(const int64_t* seeds, int64_t pop, int64_t n, uint64_t offset,
                        float* out, void* stream);

/*
 * vn_noise_dump_ex -- vn_noise_dump with a choice of distribution:
 *     out[i, t] = noise_kind(seed_i, offset + t),  out [pop, n] fp32.
 * VN_NOISE_UNIFORM is bit-exact with vn_noise_dump; VN_NOISE_GAUSSIAN is the
 * Box-Muller variant within the error stated at vn_noise. Same conventions and
 * errors as vn_noise_dump; an unknown kind returns VN_ERR_VALUE.
 */
vn_status vn_noise_dump_ex(const int64_t* seeds, int64_t pop, int64_t n, uint64_t offset,
                           vn_noise kind, float* out, void* stream);

/*
 * vn_gradient_ex -- the gradient estimate over a flat range of n elements with
 * a choice of distribution:
 *     grad[e] = sum_i fitness[i] * noise_kind(seed_i, offset + e) / (pop * sigma),  e < n.
 * With VN_NOISE_UNIFORM this is vn_bias_gradient(fitness, seeds, pop, n, ...)
 * (and a weight block's gradient is the same range, row-major). Same
 * conventions and errors as vn_weight_gradient; an unknown kind returns VN_ERR_VALUE.
 */
vn_status vn_gradient_ex(const float* fitness, const int64_t* seeds, int64_t pop, int64_t n,
                         double sigma, uint64_t offset, vn_noise kind, float* grad, void* stream);

/*
 * vn_gradient_update -- vn_gradient_ex and vn_es_update in one launch: the
 * gradient estimate over a flat range of n parameters and the ES step on it,
 *     grad[e]  = sum_i fitness[i] * noise_kind(seed_i, offset + e) / (pop * sigma)
 *     theta[e] = fma(lr, grad[e], theta[e])                      (fp32, in place)
 * for e < n (the module description's estimate, ascended with step lr). grad and
 * theta are both bit-identical to vn_gradient_ex followed by vn_es_update(theta,
 * grad, n, lr). theta [n] fp32, 4-byte aligned, must not overlap grad, fitness
 * or seeds; lr finite. Other arguments, conventions and errors as vn_gradient_ex.
 */
vn_status vn_gradient_update(const float* fitness, const int64_t* seeds, int64_t pop, int64_t n,
                             double sigma, uint64_t offset, vn_noise kind, double lr, float* grad,
                             float* theta, void* stream);

/*
 * vn_reduce_metric -- "virtual_reduce_metric" (API entry of the page):
 *     fitness[i] = mean_k | center[k] + sigma * PRNG(seed_i, offset + k) |
 * center [n_params] fp32, seeds [pop] int64, fitness [pop] fp32. n_params >= 1;
 * sigma finite. The sum over k is accumulated in fp32 in a fixed order and
 * multiplied by fp32(1 / n_params).
 */
vn_status vn_reduce_metric(const float* center, const int64_t* seeds, int64_t pop,
                           int64_t n_params, double sigma, uint64_t offset,
                           float* fitness, void* stream);

/*
 * vn_perturbed_mlp -- a chain of "virtual_perturbed_linear" layers (API entry
 * of the page) evaluated in one launch, for ES policies:
 *     h_0 = X[i];  h_{l+1} = act_l( h_l @ (W_l + sigma*N_{i,l})^T + (b_l + sigma*nb_{i,l}) )
 *     Y[i] = h_{n_layers}
 * act_l = `act` for every layer but the last, which has none. Layer l reads its
 * weight noise at offsets[l] + j*in_l + k and its bias noise at
 * offsets[l] + out_l*in_l + j, exactly as vn_perturbed_linear with offset =
 * offsets[l] would (with "compute_offsets" over (W_0, b_0, W_1, b_1, ...) the
 * weight offsets are entries 0, 2, 4, ...).
 * n_layers  1 .. 8.
 * dims      HOST array of n_layers + 1 sizes: in_0, out_0 (= in_1), ..., out_{n-1}.
 * w         HOST array of n_layers DEVICE pointers, w[l] fp32 [dims[l+1], dims[l]].
 * b         HOST array of n_layers DEVICE pointers, b[l] fp32 [dims[l+1]] or NULL
 *           (no bias and no bias noise for that layer); b itself may be NULL
 *           (no layer has a bias).
 * offsets   HOST array of n_layers weight-block offsets.
 * x         [pop, batch, dims[0]] of x_dt (VN_F32 or VN_BF16), or [batch, dims[0]]
 *           when x_shared != 0.      y  [pop, batch, dims[n_layers]] fp32.
 * batch     0 .. 8 (the per-individual batch of a policy rollout); larger
 *           batches return VN_ERR_SHAPE (use vn_perturbed_linear per layer).
 * Arithmetic is fp32 throughout (as the FFMA path of vn_perturbed_linear); the
 * activations between layers stay on chip. Layers wider than the device's
 * shared memory allows for one individual (about 3,600 units at batch 8, far
 * more at batch 1) return VN_ERR_SHAPE.
 */
vn_status vn_perturbed_mlp(const void* x, vn_dtype x_dt, int x_shared,
                           int64_t n_layers, const int64_t* dims,
                           const float* const* w, const float* const* b,
                           const uint64_t* offsets,
                           const int64_t* seeds, int64_t pop, int64_t batch,
                           double sigma, vn_act act, float* y, void* stream);

/*
 * vn_perturbed_mlp_ex -- vn_perturbed_mlp with a choice of noise distribution:
 * every N_{i,l} and nb_{i,l} is noise_kind(seed_i, index) at the same indices
 * (VN_NOISE_UNIFORM: vn_perturbed_mlp exactly; VN_NOISE_GAUSSIAN: the Box-Muller
 * variant of vn_noise, within its stated error, so that a Gaussian ES generation
 * pairs this forward with vn_gradient_ex / vn_gradient_update of the same kind).
 * With n_layers = 1 it is the single perturbed linear (fp32 W, batch <= 8) with
 * either noise. Same arguments, conventions and errors as vn_perturbed_mlp; an
 * unknown kind returns VN_ERR_VALUE.
 */
vn_status vn_perturbed_mlp_ex(const void* x, vn_dtype x_dt, int x_shared,
                              int64_t n_layers, const int64_t* dims,
                              const float* const* w, const float* const* b,
                              const uint64_t* offsets,
                              const int64_t* seeds, int64_t pop, int64_t batch,
                              double sigma, vn_act act, vn_noise kind, float* y, void* stream);

/*
 * vn_centered_ranks -- fitness shaping by centered ranks, the "fitness =
 * centered ranks in [-0.5, 0.5]" of the ES policy workload (the page's
 * gradient entries take the shaped fitness as given):
 *     out[i] = rank_i / (pop - 1) - 0.5      (out[0] = -0.5 when pop == 1)
 * rank_i = number of j with fitness[j] < fitness[i], plus the number of j < i
 * with an equal value: ascending order, ties by index. The comparison is a
 * total order on the float bit patterns (-0 below +0; NaNs beyond the
 * infinities on their sign's side), so the ranks are a permutation of
 * 0..pop-1 and out a permutation of {r / (pop - 1) - 0.5}. rank_i is converted
 * to fp32 with round-to-nearest-even before the division: exact up to 2^24
 * individuals, rounded above. fitness and out are fp32 [pop], 4-byte aligned,
 * and must not overlap. 0 <= pop < 2^31. The work is pop^2 comparisons.
 */
vn_status vn_centered_ranks(const float* fitness, int64_t pop, float* out, void* stream);

/*
 * vn_es_update -- the ES parameter step on a flat parameter vector:
 *     theta[k] = fma(lr, grad[k], theta[k]),  k < n   (fp32, in place)
 * With grad from vn_weight_gradient / vn_bias_gradient over the blocks laid out
 * by compute_offsets, lr > 0 ascends the fitness. lr finite; theta and grad
 * fp32, 4-byte aligned (16-byte alignment of both takes a vector path), and
 * must not overlap.
 */
vn_status vn_es_update(float* theta, const float* grad, int64_t n, double lr, void* stream);

/* Synchronises `stream`, then reads and clears the current device's status
 * word: VN_ERR_TIMEOUT if a kernel of this library recorded an expired wait
 * since the last call, VN_ERR_CUDA if synchronisation failed, else VN_OK. */
vn_status vn_device_status(void* stream);

/*
 * vn_hash_probe -- a measurement kernel, not a step of the method: the noise
 * hash and nothing else,
 *     sums[t] = sum_{e < m} PRNG(seed, offset + t*m + e),  t < n_sums,
 * accumulated in fp32 as two partial sums, over the even e and over the odd e
 * (each in order of e), added at the end (PRNG as defined at the top of this file).
 * One thread per t regenerates its m elements in registers and writes one
 * float, so the launch time is the hash's own: its element rate is the
 * measured ceiling of the integer ALU pipe for this hash, against which the
 * other kernels' rates can be read. sums [n_sums] fp32, 4-byte aligned;
 * 0 <= n_sums <= 2^31, m >= 0, n_sums * m < 2^63.
 */
vn_status vn_hash_probe(int64_t seed, uint64_t offset, int64_t n_sums, int64_t m, float* sums,
                        void* stream);

/* Test hook for the bounded-wait machinery of the tensor-core kernel; not part
 * of the method. Runs the tensor-core forward with the arguments of
 * vn_perturbed_linear (the same checks, with the real pop; VN_PATH_TC) but with every
 * barrier wait limited to `timeout_ms` (0 < timeout_ms <= 60000) and one
 * hashing thread of the first CTA skipping its arrive at stage
 * `withhold_stage` (>= 0), so that the MMA thread's wait on that stage can
 * never complete. The kernel must record VN_ERR_TIMEOUT in the status word,
 * stop every role, wait (bounded) for its copies and MMAs in flight, free its
 * tensor memory and return; vn_device_status() then reports VN_ERR_TIMEOUT and
 * the context stays usable. y is left partly unwritten. No GPU fault, trap or
 * hang is involved. If the CTA has fewer stages than withhold_stage, nothing is
 * withheld and the call completes normally. The hook exists for bf16 W and Y
 * only (VN_ERR_DTYPE otherwise) and needs a nonempty output (VN_ERR_SHAPE). */
vn_status vn_testhook_linear_tc_withhold(const void* x, vn_dtype x_dt, int x_shared,
                                         const void* w, vn_dtype w_dt,
                                         const void* b, vn_dtype b_dt,
                                         const int64_t* seeds, int64_t pop, int64_t batch,
                                         int64_t in, int64_t out, double sigma, uint64_t offset,
                                         void* y, vn_dtype y_dt, int64_t withhold_stage,
                                         double timeout_ms, void* stream);

/* A static, human-readable name for a status code. */
const char* vn_status_string(vn_status status);

/* The CUDA error text behind the calling thread's last VN_ERR_CUDA ("" if none). */
const char* vn_last_error_message(void);

/* The forward path vn_perturbed_linear would take for these arguments on the
 * current device (VN_PATH_FFMA or VN_PATH_TC); launches nothing. */
vn_path vn_perturbed_linear_path(const void* x, vn_dtype x_dt, int x_shared,
                                 const void* w, vn_dtype w_dt, int64_t batch,
                                 int64_t in, int64_t out);

/* ABI version: (major << 16) | minor. */
int vn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* VN_H */
