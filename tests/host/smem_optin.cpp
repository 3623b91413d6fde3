// Host-only test of vn_smem.h: the two CUDA runtime calls it makes are replaced by
// stand-ins that keep the attribute per (device, kernel), with a per-thread current
// device, so the opt-in can be checked without a GPU:
//   * one device: raised when a launch needs more, never lowered, set once per size;
//   * a second device gets its own opt-in (a single record for all devices would skip it);
//   * two kernels keep separate records;
//   * 16 threads on 4 devices: after every ensure_dynamic_smem the launch size fits.
#include <cstdio>
#include <map>
#include <mutex>
#include <random>
#include <thread>
#include <utility>
#include <vector>

#include "vn_smem.h"

namespace {
thread_local int g_device = 0;
std::mutex g_mu;
std::map<std::pair<int, const void*>, int> g_attr;
int g_sets = 0;

bool fits(const void* fn, size_t smem) {
  std::lock_guard<std::mutex> lock(g_mu);
  auto it = g_attr.find({g_device, fn});
  return smem <= 48 * 1024 || (it != g_attr.end() && static_cast<size_t>(it->second) >= smem);
}

int failures = 0;
void expect(bool ok, const char* what) {
  if (!ok) {
    std::printf("FAIL: %s\n", what);
    ++failures;
  }
}
}  // namespace

extern "C" cudaError_t cudaGetDevice(int* device) {
  *device = g_device;
  return cudaSuccess;
}

extern "C" cudaError_t cudaFuncSetAttribute(const void* fn, enum cudaFuncAttribute attr, int value) {
  if (attr != cudaFuncAttributeMaxDynamicSharedMemorySize) return cudaErrorInvalidValue;
  std::lock_guard<std::mutex> lock(g_mu);
  g_attr[{g_device, fn}] = value;  // sets, as the runtime does: a smaller value lowers it
  ++g_sets;
  return cudaSuccess;
}

int main() {
  static vn::SmemRecord rec_a, rec_b, rec_c;
  static const int kernel_a = 0, kernel_b = 0, kernel_c = 0;  // stand-in kernel addresses
  const void* a = &kernel_a;
  const void* b = &kernel_b;
  const void* c = &kernel_c;

  g_device = 0;
  expect(vn::ensure_dynamic_smem(a, 100000, rec_a) == cudaSuccess && fits(a, 100000), "first opt-in");
  expect(g_sets == 1, "one set");
  expect(vn::ensure_dynamic_smem(a, 50000, rec_a) == cudaSuccess && g_sets == 1 && fits(a, 100000),
         "a smaller size neither sets nor lowers");
  expect(vn::ensure_dynamic_smem(a, 200000, rec_a) == cudaSuccess && g_sets == 2 && fits(a, 200000),
         "a larger size raises it");
  expect(vn::ensure_dynamic_smem(a, 200000, rec_a) == cudaSuccess && g_sets == 2, "the same size: no set");

  g_device = 1;
  expect(!fits(a, 100000), "device 1 starts without the opt-in");
  expect(vn::ensure_dynamic_smem(a, 100000, rec_a) == cudaSuccess && fits(a, 100000) && g_sets == 3,
         "device 1 gets its own opt-in");
  expect(vn::ensure_dynamic_smem(b, 150000, rec_b) == cudaSuccess && fits(b, 150000) && fits(a, 100000),
         "a second kernel keeps its own record");

  std::vector<std::thread> threads;
  int thread_failures[16] = {};
  for (int t = 0; t < 16; ++t) {
    threads.emplace_back([t, c, &thread_failures] {
      std::mt19937 rng(1234 + t);
      for (int k = 0; k < 4000; ++k) {
        g_device = static_cast<int>(rng() % 4);
        const size_t smem = 49152 + 1024 * (rng() % 180);
        if (vn::ensure_dynamic_smem(c, smem, rec_c) != cudaSuccess || !fits(c, smem))
          ++thread_failures[t];
      }
    });
  }
  for (auto& th : threads) th.join();
  int conc = 0;
  for (int t = 0; t < 16; ++t) conc += thread_failures[t];
  expect(conc == 0, "every size fits right after its opt-in, across 16 threads and 4 devices");

  g_device = vn::kMaxDevices;
  expect(vn::ensure_dynamic_smem(a, 100000, rec_a) == cudaErrorInvalidDevice, "device index past the record");

  if (failures == 0) std::printf("ok\n");
  return failures == 0 ? 0 : 1;
}
