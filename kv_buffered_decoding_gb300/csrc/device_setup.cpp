// Per-device launch set-up shared by every launcher.
//
// A kernel's dynamic shared-memory limit (cudaFuncSetAttribute) and its
// occupancy are properties of one device: a process that drives several GPUs,
// one pool per GPU, has to configure each of them.  Both helpers act on the
// current device and cache their answer per (device, kernel) behind one mutex,
// so launches from several host threads are safe and each device is configured
// once.
#include <atomic>
#include <cstdint>
#include <map>
#include <mutex>
#include <utility>

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime_api.h>

#include "kvb_internal.h"

namespace kvb {
namespace {

std::mutex g_mu;
std::map<std::pair<int, const void *>, size_t> g_smem;  // configured dynamic smem bytes
std::map<std::pair<std::pair<int, const void *>, std::pair<int, size_t>>, int> g_ctas;
std::atomic<int> g_prefill_polls{0};

}  // namespace

cudaError_t ensure_smem(const void *kernel, size_t bytes) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(g_mu);
  size_t &have = g_smem[{dev, kernel}];
  if (bytes <= have) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e != cudaSuccess) return e;
  have = bytes;
  return cudaSuccess;
}

cudaError_t resident_ctas(const void *kernel, int threads, size_t smem, int *out) {
  *out = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    auto it = g_ctas.find({{dev, kernel}, {threads, smem}});
    if (it != g_ctas.end()) {
      *out = it->second;
      return cudaSuccess;
    }
  }
  if ((e = ensure_smem(kernel, smem)) != cudaSuccess) return e;
  int sms = 0, per_sm = 0;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, smem)) != cudaSuccess)
    return e;
  std::lock_guard<std::mutex> lock(g_mu);
  g_ctas[{{dev, kernel}, {threads, smem}}] = sms * per_sm;
  *out = sms * per_sm;
  return cudaSuccess;
}

cudaError_t sm_count(int *out) {
  *out = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  return cudaDeviceGetAttribute(out, cudaDevAttrMultiProcessorCount, dev);
}

namespace {
// the driver's tensor-map encoder, looked up once (null when unavailable)
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return encode;
}
}  // namespace

cudaError_t encode_state_map(StateMap *out, float *state, uint64_t rows) {
  static_assert(sizeof(StateMap) == sizeof(CUtensorMap) && alignof(StateMap) >= 64, "tensor map");
  const PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
  if (!encode || !state || rows == 0 || rows > (1ull << 31)) return cudaErrorNotSupported;
  const cuuint64_t dims[2] = {128, rows};
  const cuuint64_t strides[1] = {128 * sizeof(float)};
  const cuuint32_t box[2] = {32, 128};
  const cuuint32_t elem[2] = {1, 1};
  CUresult r = encode(reinterpret_cast<CUtensorMap *>(out), CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, state, dims,
                      strides, box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B_ATOM_32B,
                      CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorNotSupported;
}

cudaError_t encode_prefill_maps(PrefillMaps *out, const TokenIO &io, int Hk, int Hv) {
  static_assert(sizeof(TmaMap) == sizeof(CUtensorMap) && alignof(TmaMap) >= 64, "tensor map");
  const PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
  const uint64_t tokens = (uint64_t)(io.nrows > 0 ? io.nrows : 0) * (uint64_t)(io.T > 0 ? io.T : 0);
  if (!encode || tokens == 0 || tokens >= (1ull << 31) || Hk <= 0 || Hv <= 0) return cudaErrorNotSupported;
  auto one = [&](TmaMap *m, const void *base, int heads, cuuint32_t box0, CUtensorMapSwizzle sw, bool f32) {
    if (!base || (reinterpret_cast<uintptr_t>(base) & 15) != 0) return false;
    const cuuint64_t esz = f32 ? 4 : 2;
    const cuuint64_t dims[3] = {128, (cuuint64_t)heads, tokens};
    const cuuint64_t strides[2] = {128 * esz, (cuuint64_t)heads * 128 * esz};  // bytes
    const cuuint32_t box[3] = {box0, 1, 64};
    const cuuint32_t elem[3] = {1, 1, 1};
    return encode(reinterpret_cast<CUtensorMap *>(m),
                  f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                  const_cast<void *>(base), dims, strides, box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
  };
  const bool ok = one(&out->q, io.q, Hk, 64, CU_TENSOR_MAP_SWIZZLE_128B, false) &&
                  one(&out->k, io.k, Hk, 64, CU_TENSOR_MAP_SWIZZLE_128B, false) &&
                  one(&out->v, io.v, Hv, 128, CU_TENSOR_MAP_SWIZZLE_NONE, false) &&
                  one(&out->o, io.o, Hv, 128, CU_TENSOR_MAP_SWIZZLE_NONE, true);
  return ok ? cudaSuccess : cudaErrorNotSupported;
}

int prefill_first_wait_polls() { return g_prefill_polls.load(std::memory_order_relaxed); }
void set_prefill_first_wait_polls(int polls) { g_prefill_polls.store(polls, std::memory_order_relaxed); }

}  // namespace kvb
