// vn_api.cu -- the C ABI declared in include/vn.h: host-side validation,
// path selection and launch. Every argument is checked here, before anything
// touches the device; a failing check returns its status and launches nothing.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdio>
#include <mutex>

#include "vn.h"
#include "vn_internal.h"

namespace vn {

cudaError_t device_info(DeviceInfo* info) {
  static DeviceInfo cache[kMaxDevices];
  static std::mutex mu;
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  DeviceInfo& c = cache[dev];
  if (c.device != dev) {
    DeviceInfo d;
    d.device = dev;
    if ((err = cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess ||
        (err = cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
        (err = cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
        (err = cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) != cudaSuccess)
      return err;
    c = d;
  }
  *info = c;
  return cudaSuccess;
}

}  // namespace vn

namespace {

thread_local char g_last_error[256] = "";

vn_status cuda_failure(cudaError_t err) {
  std::snprintf(g_last_error, sizeof(g_last_error), "%s: %s", cudaGetErrorName(err),
                cudaGetErrorString(err));
  return VN_ERR_CUDA;
}

vn_status launched(cudaError_t err) { return err == cudaSuccess ? VN_OK : cuda_failure(err); }

bool dtype_ok(vn_dtype d) { return d == VN_F32 || d == VN_BF16; }
size_t dtype_size(vn_dtype d) { return d == VN_BF16 ? 2 : 4; }
bool aligned(const void* p, size_t a) { return reinterpret_cast<uintptr_t>(p) % a == 0; }

// r = a * b, false when it does not fit in int64 (inputs are >= 0).
bool mul(int64_t a, int64_t b, int64_t* r) { return !__builtin_mul_overflow(a, b, r); }

// The byte ranges [p, p + pb) and [q, q + qb) share a byte (an empty range shares none).
bool overlap(const void* p, int64_t pb, const void* q, int64_t qb) {
  if (p == nullptr || q == nullptr || pb <= 0 || qb <= 0) return false;
  const uintptr_t a = reinterpret_cast<uintptr_t>(p), b = reinterpret_cast<uintptr_t>(q);
  return a < b + static_cast<uintptr_t>(qb) && b < a + static_cast<uintptr_t>(pb);
}

bool float_sigma(double sigma, float* out) {
  if (!std::isfinite(sigma)) return false;
  const float f = static_cast<float>(sigma);
  if (!std::isfinite(f)) return false;
  *out = f;
  return true;
}

bool device_is_cc10(const vn::DeviceInfo& d) { return d.cc_major == 10; }

// VN_PATH_AUTO takes the tensor-core path from this per-individual batch on:
// below it the MMA's N of 16 would be mostly padding.
constexpr int64_t kAutoTcMinBatch = 16;

// The checks of a perturbed linear call (vn_perturbed_linear_kind and the test
// hook share them): dtypes, enums, sizes, sigma, size products, nulls,
// alignment and overlaps, in that order. On VN_OK, *empty tells whether the
// output has no elements (nothing to launch) and *a holds the arguments.
vn_status check_linear(const void* x, vn_dtype x_dt, int x_shared, const void* w, vn_dtype w_dt,
                       const void* b, vn_dtype b_dt, const int64_t* seeds, int64_t pop,
                       int64_t batch, int64_t in, int64_t out, double sigma, uint64_t offset,
                       void* y, vn_dtype y_dt, vn_act act, vn_noise kind, vn::LinearArgs* a,
                       bool* empty) {
  if (kind != VN_NOISE_UNIFORM && kind != VN_NOISE_GAUSSIAN) return VN_ERR_VALUE;
  if (!dtype_ok(x_dt) || !dtype_ok(w_dt) || (b != nullptr && !dtype_ok(b_dt)) || !dtype_ok(y_dt))
    return VN_ERR_DTYPE;
  const vn_dtype want_y = (x_dt == VN_BF16 && w_dt == VN_BF16) ? VN_BF16 : VN_F32;
  if (y_dt != want_y) return VN_ERR_DTYPE;
  if (act != VN_ACT_NONE && act != VN_ACT_TANH) return VN_ERR_VALUE;
  if (pop < 0 || batch < 0 || in < 0 || out < 0) return VN_ERR_SHAPE;
  float sig;
  if (!float_sigma(sigma, &sig)) return VN_ERR_VALUE;
  int64_t x_elems, y_elems, w_elems, t;
  if (!mul(batch, in, &x_elems) || (!x_shared && !mul(x_elems, pop, &x_elems)) ||
      !mul(pop, batch, &t) || !mul(t, out, &y_elems) || !mul(out, in, &w_elems))
    return VN_ERR_OVERFLOW;
  *empty = y_elems == 0;
  if (*empty) return VN_OK;
  if (seeds == nullptr || y == nullptr || (x_elems > 0 && x == nullptr) ||
      (w_elems > 0 && w == nullptr))
    return VN_ERR_NULL;
  if (!aligned(seeds, 8) || !aligned(y, dtype_size(y_dt)) || !aligned(x, dtype_size(x_dt)) ||
      !aligned(w, dtype_size(w_dt)) || (b != nullptr && !aligned(b, dtype_size(b_dt))))
    return VN_ERR_ALIGN;
  int64_t yb, xb, wb, bb, sb;
  if (!mul(y_elems, dtype_size(y_dt), &yb) || !mul(x_elems, dtype_size(x_dt), &xb) ||
      !mul(w_elems, dtype_size(w_dt), &wb) || !mul(out, dtype_size(b_dt), &bb) ||
      !mul(pop, 8, &sb))
    return VN_ERR_OVERFLOW;
  if (overlap(y, yb, x, xb) || overlap(y, yb, w, wb) || overlap(y, yb, b, bb) ||
      overlap(y, yb, seeds, sb))
    return VN_ERR_VALUE;
  a->x = x; a->x_dt = x_dt; a->x_shared = x_shared ? 1 : 0;
  a->w = w; a->w_dt = w_dt; a->b = b; a->b_dt = b_dt;
  a->seeds = seeds; a->pop = pop; a->batch = batch; a->in = in; a->out = out;
  a->sigma = sig; a->offset = offset; a->y = y; a->y_dt = y_dt; a->act = act; a->kind = kind;
  return VN_OK;
}

}  // namespace

extern "C" {

const char* vn_status_string(vn_status s) {
  switch (s) {
    case VN_OK: return "VN_OK";
    case VN_ERR_NULL: return "VN_ERR_NULL: a required pointer is NULL";
    case VN_ERR_SHAPE: return "VN_ERR_SHAPE: invalid size";
    case VN_ERR_DTYPE: return "VN_ERR_DTYPE: unsupported dtype or dtype combination";
    case VN_ERR_VALUE: return "VN_ERR_VALUE: invalid value (sigma, enum)";
    case VN_ERR_ALIGN: return "VN_ERR_ALIGN: pointer not aligned to its element size";
    case VN_ERR_OVERFLOW: return "VN_ERR_OVERFLOW: size product does not fit in int64";
    case VN_ERR_TIMEOUT: return "VN_ERR_TIMEOUT: a device-side bounded wait ran out";
    case VN_ERR_CUDA: return "VN_ERR_CUDA: a CUDA runtime call failed";
    case VN_ERR_DEVICE: return "VN_ERR_DEVICE: this path needs a compute capability 10.x GPU";
    case VN_ERR_PATH: return "VN_ERR_PATH: the forced path cannot run these arguments";
  }
  return "unknown vn_status";
}

const char* vn_last_error_message(void) { return g_last_error; }

int vn_version(void) { return (1 << 16) | 0; }

vn_status vn_noise_dump(const int64_t* seeds, int64_t pop, int64_t n, uint64_t offset,
                        float* out, void* stream) {
  return vn_noise_dump_ex(seeds, pop, n, offset, VN_NOISE_UNIFORM, out, stream);
}

vn_status vn_noise_dump_ex(const int64_t* seeds, int64_t pop, int64_t n, uint64_t offset,
                           vn_noise kind, float* out, void* stream) {
  if (kind != VN_NOISE_UNIFORM && kind != VN_NOISE_GAUSSIAN) return VN_ERR_VALUE;
  if (pop < 0 || n < 0) return VN_ERR_SHAPE;
  int64_t total;
  if (!mul(pop, n, &total)) return VN_ERR_OVERFLOW;
  if (total == 0) return VN_OK;
  if (seeds == nullptr || out == nullptr) return VN_ERR_NULL;
  if (!aligned(seeds, 8) || !aligned(out, 4)) return VN_ERR_ALIGN;
  int64_t out_bytes, seed_bytes;
  if (!mul(total, 4, &out_bytes) || !mul(pop, 8, &seed_bytes)) return VN_ERR_OVERFLOW;
  if (overlap(out, out_bytes, seeds, seed_bytes)) return VN_ERR_VALUE;
  return launched(vn::launch_noise_dump(seeds, pop, n, offset, kind, out,
                                        static_cast<cudaStream_t>(stream)));
}

static vn_status gradient(const float* fitness, const int64_t* seeds, int64_t pop, int64_t m_rows,
                          int64_t m_cols, double sigma, uint64_t offset, vn_noise kind,
                          float* grad, void* stream, float* theta = nullptr, double lr = 0.0) {
  if (kind != VN_NOISE_UNIFORM && kind != VN_NOISE_GAUSSIAN) return VN_ERR_VALUE;
  if (pop < 1 || m_rows < 0 || m_cols < 0) return VN_ERR_SHAPE;
  int64_t m;
  if (!mul(m_rows, m_cols, &m)) return VN_ERR_OVERFLOW;
  float sig;
  if (!float_sigma(sigma, &sig) || sig == 0.f) return VN_ERR_VALUE;
  const double inv = 1.0 / (static_cast<double>(pop) * sigma);
  const float scale = static_cast<float>(inv);
  if (!std::isfinite(scale) || scale == 0.f) return VN_ERR_VALUE;
  float lr_f = 0.f;
  if (theta != nullptr && !float_sigma(lr, &lr_f)) return VN_ERR_VALUE;
  if (m == 0) return VN_OK;
  if (fitness == nullptr || seeds == nullptr || grad == nullptr) return VN_ERR_NULL;
  if (!aligned(fitness, 4) || !aligned(seeds, 8) || !aligned(grad, 4)) return VN_ERR_ALIGN;
  if (theta != nullptr && !aligned(theta, 4)) return VN_ERR_ALIGN;
  int64_t m_bytes, seed_bytes;
  if (!mul(m, 4, &m_bytes) || !mul(pop, 8, &seed_bytes)) return VN_ERR_OVERFLOW;
  const int64_t fit_bytes = pop * 4;
  // The outputs (grad, and theta when given) may not share memory with an input or each other.
  if (overlap(grad, m_bytes, fitness, fit_bytes) || overlap(grad, m_bytes, seeds, seed_bytes))
    return VN_ERR_VALUE;
  if (theta != nullptr &&
      (overlap(theta, m_bytes, grad, m_bytes) || overlap(theta, m_bytes, fitness, fit_bytes) ||
       overlap(theta, m_bytes, seeds, seed_bytes)))
    return VN_ERR_VALUE;
  return launched(vn::launch_grad(fitness, seeds, pop, m, offset, scale, kind, grad,
                                  static_cast<cudaStream_t>(stream), theta, lr_f));
}

vn_status vn_weight_gradient(const float* fitness, const int64_t* seeds, int64_t pop,
                             int64_t out, int64_t in, double sigma, uint64_t offset,
                             float* grad_w, void* stream) {
  return gradient(fitness, seeds, pop, out, in, sigma, offset, VN_NOISE_UNIFORM, grad_w, stream);
}

vn_status vn_bias_gradient(const float* fitness, const int64_t* seeds, int64_t pop,
                           int64_t out, double sigma, uint64_t offset, float* grad_b,
                           void* stream) {
  return gradient(fitness, seeds, pop, out, 1, sigma, offset, VN_NOISE_UNIFORM, grad_b, stream);
}

vn_status vn_gradient_ex(const float* fitness, const int64_t* seeds, int64_t pop, int64_t n,
                         double sigma, uint64_t offset, vn_noise kind, float* grad, void* stream) {
  return gradient(fitness, seeds, pop, n, 1, sigma, offset, kind, grad, stream);
}

vn_status vn_gradient_update(const float* fitness, const int64_t* seeds, int64_t pop, int64_t n,
                             double sigma, uint64_t offset, vn_noise kind, double lr, float* grad,
                             float* theta, void* stream) {
  if (n > 0 && theta == nullptr) return VN_ERR_NULL;
  if (theta == nullptr) {  // n == 0: validate as the plain estimate does, launch nothing
    float lr_f;
    if (!float_sigma(lr, &lr_f)) return VN_ERR_VALUE;
    return gradient(fitness, seeds, pop, n, 1, sigma, offset, kind, grad, stream);
  }
  return gradient(fitness, seeds, pop, n, 1, sigma, offset, kind, grad, stream, theta, lr);
}

vn_status vn_reduce_metric(const float* center, const int64_t* seeds, int64_t pop,
                           int64_t n_params, double sigma, uint64_t offset, float* fitness,
                           void* stream) {
  if (pop < 0 || n_params < 1) return VN_ERR_SHAPE;
  float sig;
  if (!float_sigma(sigma, &sig)) return VN_ERR_VALUE;
  int64_t total;
  if (!mul(pop, n_params, &total)) return VN_ERR_OVERFLOW;
  if (pop == 0) return VN_OK;
  if (center == nullptr || seeds == nullptr || fitness == nullptr) return VN_ERR_NULL;
  if (!aligned(center, 4) || !aligned(seeds, 8) || !aligned(fitness, 4)) return VN_ERR_ALIGN;
  int64_t center_bytes, seed_bytes;
  if (!mul(n_params, 4, &center_bytes) || !mul(pop, 8, &seed_bytes)) return VN_ERR_OVERFLOW;
  const int64_t fit_bytes = pop * 4;  // fits: pop * 8 does
  if (overlap(fitness, fit_bytes, center, center_bytes) || overlap(fitness, fit_bytes, seeds, seed_bytes))
    return VN_ERR_VALUE;
  const float inv_n = static_cast<float>(1.0 / static_cast<double>(n_params));
  return launched(vn::launch_reduce_metric(center, seeds, pop, n_params, sig, inv_n, offset,
                                           fitness, static_cast<cudaStream_t>(stream)));
}

vn_path vn_perturbed_linear_path(const void* x, vn_dtype x_dt, int x_shared, const void* w,
                                 vn_dtype w_dt, int64_t batch, int64_t in, int64_t out) {
  (void)x_shared;
  vn::DeviceInfo dev;
  if (vn::device_info(&dev) != cudaSuccess || !device_is_cc10(dev)) return VN_PATH_FFMA;
  return (batch >= kAutoTcMinBatch && vn::linear_tc_applies(x, x_dt, w, w_dt, batch, in, out))
             ? VN_PATH_TC
             : VN_PATH_FFMA;
}

vn_status vn_perturbed_linear_ex(const void* x, vn_dtype x_dt, int x_shared, const void* w,
                                 vn_dtype w_dt, const void* b, vn_dtype b_dt,
                                 const int64_t* seeds, int64_t pop, int64_t batch, int64_t in,
                                 int64_t out, double sigma, uint64_t offset, void* y,
                                 vn_dtype y_dt, vn_path path, vn_act act, void* stream) {
  return vn_perturbed_linear_kind(x, x_dt, x_shared, w, w_dt, b, b_dt, seeds, pop, batch, in, out,
                                  sigma, offset, y, y_dt, path, act, VN_NOISE_UNIFORM, stream);
}

vn_status vn_perturbed_linear_kind(const void* x, vn_dtype x_dt, int x_shared, const void* w,
                                   vn_dtype w_dt, const void* b, vn_dtype b_dt,
                                   const int64_t* seeds, int64_t pop, int64_t batch, int64_t in,
                                   int64_t out, double sigma, uint64_t offset, void* y,
                                   vn_dtype y_dt, vn_path path, vn_act act, vn_noise kind,
                                   void* stream) {
  if (path != VN_PATH_AUTO && path != VN_PATH_FFMA && path != VN_PATH_TC) return VN_ERR_PATH;
  vn::LinearArgs a;
  bool empty = false;
  const vn_status st = check_linear(x, x_dt, x_shared, w, w_dt, b, b_dt, seeds, pop, batch, in,
                                    out, sigma, offset, y, y_dt, act, kind, &a, &empty);
  if (st != VN_OK || empty) return st;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  const bool gaussian = kind == VN_NOISE_GAUSSIAN;

  if (path == VN_PATH_FFMA && !gaussian) return launched(vn::launch_linear_ffma(a, s));
  vn::DeviceInfo dev;
  cudaError_t err = vn::device_info(&dev);
  if (err != cudaSuccess) return cuda_failure(err);
  const bool tc_ok = vn::linear_tc_applies(x, x_dt, w, w_dt, batch, in, out);
  if (path == VN_PATH_TC) {
    if (!device_is_cc10(dev)) return VN_ERR_DEVICE;
    if (!tc_ok) return VN_ERR_PATH;
    return launched(vn::launch_linear_tc(a, s));
  }
  if (path == VN_PATH_AUTO && tc_ok && batch >= kAutoTcMinBatch && device_is_cc10(dev))
    return launched(vn::launch_linear_tc(a, s));
  // fp32 W (and bias), a policy-sized batch and enough individuals to give every
  // SM a group of them: the one-launch chain kernel with one layer (its
  // individuals share each loaded W chunk, which the single-layer CUDA-core
  // kernel does not), when the layer fits its shared memory. It is also the
  // CUDA-core kernel of the Gaussian kind, for any population.
  if (w_dt == VN_F32 && (b == nullptr || b_dt == VN_F32) && batch >= 1 &&
      batch <= vn::kMlpMaxBatch && (pop >= dev.sm_count || gaussian) && in < (int64_t{1} << 31) &&
      out < (int64_t{1} << 31)) {
    const int64_t dims[2] = {in, out};
    const size_t buf = vn::mlp_buffer_floats(1, dims);
    if (vn::mlp_bytes_per_individual(batch, buf) <= static_cast<size_t>(dev.smem_optin)) {
      const float* wl[1] = {static_cast<const float*>(w)};
      const float* bl[1] = {static_cast<const float*>(b)};
      const uint64_t offs[1] = {offset};
      vn::MlpArgs m;
      m.x = x; m.x_dt = x_dt; m.x_shared = x_shared ? 1 : 0;
      m.n_layers = 1;
      m.dims = dims; m.w = wl; m.b = bl; m.offsets = offs;
      m.seeds = seeds; m.pop = pop; m.batch = batch; m.sigma = a.sigma; m.act = VN_ACT_NONE;
      m.y = static_cast<float*>(y);
      m.act_last = act;
      m.kind = kind;
      return launched(vn::launch_mlp(m, s));
    }
  }
  // The single-layer CUDA-core kernel has the uniform kind only.
  if (gaussian) return VN_ERR_PATH;
  return launched(vn::launch_linear_ffma(a, s));
}

vn_status vn_perturbed_linear(const void* x, vn_dtype x_dt, int x_shared, const void* w,
                              vn_dtype w_dt, const void* b, vn_dtype b_dt, const int64_t* seeds,
                              int64_t pop, int64_t batch, int64_t in, int64_t out, double sigma,
                              uint64_t offset, void* y, vn_dtype y_dt, void* stream) {
  return vn_perturbed_linear_ex(x, x_dt, x_shared, w, w_dt, b, b_dt, seeds, pop, batch, in, out,
                                sigma, offset, y, y_dt, VN_PATH_AUTO, VN_ACT_NONE, stream);
}

vn_status vn_testhook_linear_tc_withhold(const void* x, vn_dtype x_dt, int x_shared, const void* w,
                                         vn_dtype w_dt, const void* b, vn_dtype b_dt,
                                         const int64_t* seeds, int64_t pop, int64_t batch,
                                         int64_t in, int64_t out, double sigma, uint64_t offset,
                                         void* y, vn_dtype y_dt, int64_t withhold_stage,
                                         double timeout_ms, void* stream) {
  if (!(timeout_ms > 0.0) || !(timeout_ms <= 60000.0) || withhold_stage < 0) return VN_ERR_VALUE;
  if (w_dt != VN_BF16 || y_dt != VN_BF16) return VN_ERR_DTYPE;  // the hook's one instance
  // The same checks as a forced tensor-core call, with the real population.
  vn::LinearArgs a;
  bool empty = false;
  const vn_status st = check_linear(x, x_dt, x_shared, w, w_dt, b, b_dt, seeds, pop, batch, in,
                                    out, sigma, offset, y, y_dt, VN_ACT_NONE, VN_NOISE_UNIFORM,
                                    &a, &empty);
  if (st != VN_OK) return st;
  if (empty) return VN_ERR_SHAPE;  // the hook needs a kernel to withhold an arrive in
  vn::DeviceInfo dev;
  cudaError_t err = vn::device_info(&dev);
  if (err != cudaSuccess) return cuda_failure(err);
  if (!device_is_cc10(dev)) return VN_ERR_DEVICE;
  if (!vn::linear_tc_applies(x, x_dt, w, w_dt, batch, in, out) || pop > (int64_t{1} << 31) - 1)
    return VN_ERR_PATH;
  return launched(vn::launch_linear_tc_hook(a, static_cast<cudaStream_t>(stream), withhold_stage,
                                            static_cast<unsigned long long>(timeout_ms * 1e6)));
}

vn_status vn_perturbed_mlp(const void* x, vn_dtype x_dt, int x_shared, int64_t n_layers,
                           const int64_t* dims, const float* const* w, const float* const* b,
                           const uint64_t* offsets, const int64_t* seeds, int64_t pop,
                           int64_t batch, double sigma, vn_act act, float* y, void* stream) {
  return vn_perturbed_mlp_ex(x, x_dt, x_shared, n_layers, dims, w, b, offsets, seeds, pop, batch,
                             sigma, act, VN_NOISE_UNIFORM, y, stream);
}

vn_status vn_perturbed_mlp_ex(const void* x, vn_dtype x_dt, int x_shared, int64_t n_layers,
                              const int64_t* dims, const float* const* w, const float* const* b,
                              const uint64_t* offsets, const int64_t* seeds, int64_t pop,
                              int64_t batch, double sigma, vn_act act, vn_noise kind, float* y,
                              void* stream) {
  if (kind != VN_NOISE_UNIFORM && kind != VN_NOISE_GAUSSIAN) return VN_ERR_VALUE;
  if (!dtype_ok(x_dt)) return VN_ERR_DTYPE;
  if (act != VN_ACT_NONE && act != VN_ACT_TANH) return VN_ERR_VALUE;
  if (n_layers < 1 || n_layers > vn::kMlpMaxLayers) return VN_ERR_SHAPE;
  if (dims == nullptr || w == nullptr || offsets == nullptr) return VN_ERR_NULL;
  if (pop < 0 || batch < 0 || batch > vn::kMlpMaxBatch) return VN_ERR_SHAPE;
  constexpr int64_t kMaxDim = (int64_t{1} << 31) - 1;
  for (int64_t l = 0; l <= n_layers; ++l)
    if (dims[l] < 0 || dims[l] > kMaxDim) return VN_ERR_SHAPE;
  float sig;
  if (!float_sigma(sigma, &sig)) return VN_ERR_VALUE;
  int64_t x_elems, y_elems, t;
  if (!mul(batch, dims[0], &x_elems) || (!x_shared && !mul(x_elems, pop, &x_elems)) ||
      !mul(pop, batch, &t) || !mul(t, dims[n_layers], &y_elems))
    return VN_ERR_OVERFLOW;
  for (int64_t l = 0; l < n_layers; ++l) {
    int64_t we;
    if (!mul(dims[l], dims[l + 1], &we)) return VN_ERR_OVERFLOW;
    if (we > 0 && w[l] == nullptr) return VN_ERR_NULL;
    if (!aligned(w[l], 4) || (b != nullptr && !aligned(b[l], 4))) return VN_ERR_ALIGN;
  }
  if (y_elems == 0) return VN_OK;
  if (seeds == nullptr || y == nullptr || (x_elems > 0 && x == nullptr)) return VN_ERR_NULL;
  if (!aligned(seeds, 8) || !aligned(y, 4) || !aligned(x, dtype_size(x_dt))) return VN_ERR_ALIGN;
  {
    int64_t yb, xb, sb;
    if (!mul(y_elems, 4, &yb) || !mul(x_elems, dtype_size(x_dt), &xb) || !mul(pop, 8, &sb))
      return VN_ERR_OVERFLOW;
    if (overlap(y, yb, x, xb) || overlap(y, yb, seeds, sb)) return VN_ERR_VALUE;
    for (int64_t l = 0; l < n_layers; ++l) {
      int64_t wb;
      if (!mul(dims[l] * dims[l + 1], 4, &wb)) return VN_ERR_OVERFLOW;  // the product fits: checked above
      if (overlap(y, yb, w[l], wb) || (b != nullptr && overlap(y, yb, b[l], dims[l + 1] * 4)))
        return VN_ERR_VALUE;
    }
  }
  // The one device-dependent check: both activation buffers of one individual
  // must fit in the device's shared memory.
  const size_t buf = vn::mlp_buffer_floats(static_cast<int>(n_layers), dims);
  vn::DeviceInfo dev;
  cudaError_t err = vn::device_info(&dev);
  if (err != cudaSuccess) return cuda_failure(err);
  if (vn::mlp_bytes_per_individual(batch, buf) > static_cast<size_t>(dev.smem_optin))
    return VN_ERR_SHAPE;

  static const float* const kNoBias[vn::kMlpMaxLayers] = {};
  vn::MlpArgs m;
  m.x = x; m.x_dt = x_dt; m.x_shared = x_shared ? 1 : 0;
  m.n_layers = static_cast<int>(n_layers);
  m.dims = dims; m.w = w; m.b = b != nullptr ? b : kNoBias; m.offsets = offsets;
  m.seeds = seeds; m.pop = pop; m.batch = batch; m.sigma = sig; m.act = act; m.y = y;
  m.kind = kind;
  return launched(vn::launch_mlp(m, static_cast<cudaStream_t>(stream)));
}

vn_status vn_centered_ranks(const float* fitness, int64_t pop, float* out, void* stream) {
  if (pop < 0 || pop > (int64_t{1} << 31) - 1) return VN_ERR_SHAPE;
  if (pop == 0) return VN_OK;
  if (fitness == nullptr || out == nullptr) return VN_ERR_NULL;
  if (!aligned(fitness, 4) || !aligned(out, 4)) return VN_ERR_ALIGN;
  if (overlap(out, pop * 4, fitness, pop * 4)) return VN_ERR_VALUE;  // pop < 2^31: no overflow
  return launched(vn::launch_centered_ranks(fitness, pop, out, static_cast<cudaStream_t>(stream)));
}

vn_status vn_es_update(float* theta, const float* grad, int64_t n, double lr, void* stream) {
  if (n < 0) return VN_ERR_SHAPE;
  float lr_f;
  if (!float_sigma(lr, &lr_f)) return VN_ERR_VALUE;
  if (n == 0) return VN_OK;
  if (theta == nullptr || grad == nullptr) return VN_ERR_NULL;
  if (!aligned(theta, 4) || !aligned(grad, 4)) return VN_ERR_ALIGN;
  int64_t bytes;
  if (!mul(n, 4, &bytes)) return VN_ERR_OVERFLOW;
  if (overlap(theta, bytes, grad, bytes)) return VN_ERR_VALUE;
  return launched(vn::launch_es_update(theta, grad, n, lr_f, static_cast<cudaStream_t>(stream)));
}

vn_status vn_hash_probe(int64_t seed, uint64_t offset, int64_t n_sums, int64_t m, float* sums,
                        void* stream) {
  if (n_sums < 0 || n_sums > (int64_t{1} << 31) || m < 0) return VN_ERR_SHAPE;
  int64_t elems;
  if (!mul(n_sums, m, &elems)) return VN_ERR_OVERFLOW;
  if (n_sums == 0) return VN_OK;
  if (sums == nullptr) return VN_ERR_NULL;
  if (!aligned(sums, 4)) return VN_ERR_ALIGN;
  return launched(vn::launch_hash_probe(static_cast<uint64_t>(seed), offset, n_sums, m, sums,
                                        static_cast<cudaStream_t>(stream)));
}

vn_status vn_device_status(void* stream) {
  cudaError_t err = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (err != cudaSuccess) return cuda_failure(err);
  unsigned int status = 0;
  err = vn::take_device_status(&status, static_cast<cudaStream_t>(stream));
  if (err != cudaSuccess) return cuda_failure(err);
  return status ? VN_ERR_TIMEOUT : VN_OK;
}

}  // extern "C"
