// Host-side check of the per-device launch set-up (device_setup.cpp) against a
// fake CUDA runtime: the few runtime calls the helpers make are defined here, so
// the real helpers run on the CPU with a current device that the test switches.
// Prints "ok" when every check holds (test infrastructure, built by
// tests/test_device_setup.py).
#include <cstdio>
#include <map>
#include <mutex>
#include <thread>
#include <utility>
#include <vector>

#include <cuda_runtime_api.h>

#include "kvb_internal.h"

namespace {
thread_local int g_dev = 0;  // the current device, per host thread as in the runtime
std::mutex g_mu;
std::map<int, int> g_setattr;     // device -> cudaFuncSetAttribute calls
std::map<int, int> g_last_bytes;  // device -> last dynamic smem limit set
std::map<int, int> g_occupancy;   // device -> occupancy queries
}  // namespace

cudaError_t cudaGetDevice(int *device) {
  *device = g_dev;
  return cudaSuccess;
}
cudaError_t cudaFuncSetAttribute(const void *, enum cudaFuncAttribute attr, int value) {
  if (attr != cudaFuncAttributeMaxDynamicSharedMemorySize) return cudaErrorInvalidValue;
  std::lock_guard<std::mutex> lock(g_mu);
  ++g_setattr[g_dev];
  g_last_bytes[g_dev] = value;
  return cudaSuccess;
}
cudaError_t cudaDeviceGetAttribute(int *value, enum cudaDeviceAttr attr, int device) {
  if (attr != cudaDevAttrMultiProcessorCount) return cudaErrorInvalidValue;
  *value = 100 + device;  // a different SM count on every device
  return cudaSuccess;
}
cudaError_t cudaOccupancyMaxActiveBlocksPerMultiprocessor(int *num, const void *, int, size_t) {
  std::lock_guard<std::mutex> lock(g_mu);
  ++g_occupancy[g_dev];
  *num = 2;
  return cudaSuccess;
}
cudaError_t cudaGetDriverEntryPointByVersion(const char *, void **fn, unsigned int, unsigned long long,
                                             cudaDriverEntryPointQueryResult *q) {
  *fn = nullptr;
  if (q) *q = cudaDriverEntryPointSymbolNotFound;
  return cudaErrorNotSupported;
}

static int failures = 0;
#define CHECK(c)                                              \
  do {                                                        \
    if (!(c)) {                                               \
      std::printf("check failed at line %d: %s\n", __LINE__, #c); \
      ++failures;                                             \
    }                                                         \
  } while (0)

int main() {
  static const char kernel_a = 0, kernel_b = 0;  // two distinct "kernels"
  const void *ka = &kernel_a, *kb = &kernel_b;

  // device 0: the attribute is set once per (device, kernel) and raised when needed
  g_dev = 0;
  CHECK(kvb::ensure_smem(ka, 1000) == cudaSuccess);
  CHECK(kvb::ensure_smem(ka, 1000) == cudaSuccess);
  CHECK(kvb::ensure_smem(ka, 500) == cudaSuccess);
  CHECK(g_setattr[0] == 1 && g_last_bytes[0] == 1000);
  CHECK(kvb::ensure_smem(ka, 2000) == cudaSuccess);
  CHECK(g_setattr[0] == 2 && g_last_bytes[0] == 2000);
  CHECK(kvb::ensure_smem(kb, 1000) == cudaSuccess);
  CHECK(g_setattr[0] == 3);

  // device 1: the same kernel is configured again there
  g_dev = 1;
  CHECK(kvb::ensure_smem(ka, 1000) == cudaSuccess);
  CHECK(g_setattr[1] == 1 && g_last_bytes[1] == 1000);

  // resident CTAs: per device (SM count differs), queried once per device and shape
  int c0 = 0, c1 = 0, again = 0;
  g_dev = 0;
  CHECK(kvb::resident_ctas(ka, 128, 1000, &c0) == cudaSuccess);
  CHECK(kvb::resident_ctas(ka, 128, 1000, &again) == cudaSuccess);
  g_dev = 1;
  CHECK(kvb::resident_ctas(ka, 128, 1000, &c1) == cudaSuccess);
  CHECK(c0 == 200 && again == 200 && c1 == 202);
  CHECK(g_occupancy[0] == 1 && g_occupancy[1] == 1);
  int sms = 0;
  CHECK(kvb::sm_count(&sms) == cudaSuccess && sms == 101);

  // several host threads on a fresh device: configured exactly once
  std::vector<std::thread> pool;
  for (int i = 0; i < 8; ++i)
    pool.emplace_back([ka] {
      g_dev = 2;
      int out = 0;
      for (int r = 0; r < 100; ++r) {
        kvb::ensure_smem(ka, 4096);
        kvb::resident_ctas(ka, 64, 4096, &out);
      }
    });
  for (auto &t : pool) t.join();
  CHECK(g_setattr[2] == 1 && g_last_bytes[2] == 4096);
  CHECK(g_occupancy[2] >= 1);
  int c2 = 0;
  g_dev = 2;
  CHECK(kvb::resident_ctas(ka, 64, 4096, &c2) == cudaSuccess && c2 == 204);

  // the prefill wait-limit hook round-trips
  kvb::set_prefill_first_wait_polls(7);
  CHECK(kvb::prefill_first_wait_polls() == 7);
  kvb::set_prefill_first_wait_polls(0);

  if (failures == 0) std::printf("ok\n");
  return failures == 0 ? 0 : 1;
}
