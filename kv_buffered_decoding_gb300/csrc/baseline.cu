// The serving baseline KVBuffer is compared with for speculative decoding
// ("KVBuffer: IO-aware Serving for Linear Attention", Figure 2): a serving
// system with only a state pool verifies T draft tokens with the recurrent
// form, storing a temporary state after every draft; after the sampler decides
// how many drafts to accept, the request's state is replaced by the temporary
// state of the last accepted draft.
//
// verify_tempstate_kernel: per (request, value head) the state tile is read
// once into registers (the decode layout: two CTAs per head at d = 128, 16
// consecutive rows per lane) and stepped through the T drafts in registers:
//   u_j = v_j                                   (plain / gated)
//   u_j = beta_j (v_j - g_j S_{j-1}^T k_j)      (gated delta rule)
//   o_j = g_j S_{j-1}^T q_j + (q_j.k_j) u_j,    S_j = g_j S_{j-1} + k_j u_j^T
// and every S_j is written to its temporary slot: T state writes per round,
// the traffic (and memory) the buffered verify avoids.
// tempstate_accept_kernel copies temporary state j-1 into the request's slot.
#include <mutex>

#include "kvb_device.cuh"

namespace kvb {

template <typename KT, int VARIANT, int D, int NSPLIT>
__global__ void __launch_bounds__(2 * D / NSPLIT, 512 / (2 * D / NSPLIT))
    verify_tempstate_kernel(const PoolView P, const RowBatch rows, const TokenIO io,
                            float *temp) {
  constexpr int DK = D, DV = D, NT = 2 * D / NSPLIT, RPT = DK / 8, E = DK / 32;
  constexpr bool DELTA = VARIANT == kGatedDelta, GATED = VARIANT != kPlain;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int h = blockIdx.x / NSPLIT, part = blockIdx.x % NSPLIT;
  const int rsub = lane >> 2, row0 = rsub * RPT;
  const int col0 = part * (DV / NSPLIT) + warp * 16 + (lane & 3) * 4;
  const RowDesc d = rows.r[blockIdx.y];
  const size_t b = (size_t)rows.row0 + blockIdx.y;
  const int hq = h / (P.Hv / P.Hk);
  const int T = io.T;

  __shared__ __align__(16) float qs[2][DK];
  __shared__ __align__(16) float kts[2][DK];

  const float *Sp = P.state + ((size_t)d.slot * P.Hv + h) * DK * DV;
  float4 s[RPT];
#pragma unroll
  for (int j = 0; j < RPT; ++j) s[j] = ld_stream4(Sp + (row0 + j) * DV + col0);

  const KT *qg = static_cast<const KT *>(io.q) + b * T * P.Hk * DK;
  const KT *kg = static_cast<const KT *>(io.k) + b * T * P.Hk * DK;
  const KT *vg = static_cast<const KT *>(io.v) + b * T * P.Hv * DV;
  for (int j = 0; j < T; ++j) {
    const int buf = j & 1;  // double-buffered so one barrier per draft suffices
    for (int i = tid; i < DK; i += NT) {
      qs[buf][i] = P.scale * to_float(qg[((size_t)j * P.Hk + hq) * DK + i]);
      kts[buf][i] = to_float(kg[((size_t)j * P.Hk + hq) * DK + i]);
    }
    const float4 vj = ld4(vg + ((size_t)j * P.Hv + h) * DV + col0);
    const float g = GATED && io.log_g ? expf(io.log_g[(b * T + j) * P.Hv + h]) : 1.f;
    const float bj = DELTA ? io.beta[(b * T + j) * P.Hv + h] : 0.f;
    __syncthreads();
    // q_j . k_j (every warp computes it; no extra barrier)
    float qv[E], tv[E];
    load_smem<E>(&qs[buf][lane * E], qv);
    load_smem<E>(&kts[buf][lane * E], tv);
    float st = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) st = fmaf(qv[e], tv[e], st);
    st = warp_sum(st);
    // S_{j-1}^T q_j and S_{j-1}^T k_j over this lane's rows
    float4 aq = f4(0.f), ak = f4(0.f);
#pragma unroll
    for (int r = 0; r < RPT; r += 4) {
      const float4 q4 = *reinterpret_cast<const float4 *>(&qs[buf][row0 + r]);
      fma4(aq, q4.x, s[r]);
      fma4(aq, q4.y, s[r + 1]);
      fma4(aq, q4.z, s[r + 2]);
      fma4(aq, q4.w, s[r + 3]);
      if (DELTA) {
        const float4 k4 = *reinterpret_cast<const float4 *>(&kts[buf][row0 + r]);
        fma4(ak, k4.x, s[r]);
        fma4(ak, k4.y, s[r + 1]);
        fma4(ak, k4.z, s[r + 2]);
        fma4(ak, k4.w, s[r + 3]);
      }
    }
    aq = rows_sum4(aq);
    if (DELTA) ak = rows_sum4(ak);
    float4 u = vj;
    if (DELTA) {
      u.x = bj * (vj.x - g * ak.x);
      u.y = bj * (vj.y - g * ak.y);
      u.z = bj * (vj.z - g * ak.z);
      u.w = bj * (vj.w - g * ak.w);
    }
    float4 o = mul4(g, aq);
    fma4(o, st, u);
    if (rsub == 0)
      __stcs(reinterpret_cast<float4 *>(io.o + ((b * T + j) * P.Hv + h) * DV + col0), o);
    // S_j = g S_{j-1} + k_j u_j^T, stored as temporary state j
    float *Tp = temp + ((((size_t)b * T + j) * P.Hv + h) * DK) * DV;
#pragma unroll
    for (int r = 0; r < RPT; r += 4) {
      const float4 k4 = *reinterpret_cast<const float4 *>(&kts[buf][row0 + r]);
      s[r] = mul4(g, s[r]);
      s[r + 1] = mul4(g, s[r + 1]);
      s[r + 2] = mul4(g, s[r + 2]);
      s[r + 3] = mul4(g, s[r + 3]);
      fma4(s[r], k4.x, u);
      fma4(s[r + 1], k4.y, u);
      fma4(s[r + 2], k4.z, u);
      fma4(s[r + 3], k4.w, u);
    }
#pragma unroll
    for (int r = 0; r < RPT; ++r) st_stream4(Tp + (row0 + r) * DV + col0, s[r]);
  }
}

// Accept: the state of row b becomes temporary state n_acc - 1 (rows with
// n_acc = 0 are not launched).  RowDesc.n carries n_acc.
__global__ void __launch_bounds__(256) tempstate_accept_kernel(const PoolView P, const RowBatch rows,
                                                               const float *temp, int T, int DK,
                                                               int DV) {
  const RowDesc d = rows.r[blockIdx.y];
  const size_t b = (size_t)rows.row0 + blockIdx.y;
  const int h = blockIdx.x;
  const float4 *src = reinterpret_cast<const float4 *>(
      temp + ((((size_t)b * T + (d.n - 1)) * P.Hv + h) * DK) * DV);
  float4 *dst = reinterpret_cast<float4 *>(P.state + ((size_t)d.slot * P.Hv + h) * DK * DV);
  for (int i = threadIdx.x; i < DK * DV / 4; i += blockDim.x) __stcs(dst + i, __ldcs(src + i));
}

template <typename KT, int VARIANT, int D>
static cudaError_t run_tempstate(const PoolView &P, const RowBatch &rows, const TokenIO &io,
                                 float *temp, cudaStream_t s) {
  constexpr int NS = D == 128 ? 2 : 1;
  dim3 grid(P.Hv * NS, rows.count);
  verify_tempstate_kernel<KT, VARIANT, D, NS><<<grid, 2 * D / NS, 0, s>>>(P, rows, io, temp);
  return cudaGetLastError();
}

template <typename KT, int VARIANT>
static cudaError_t tempstate_d(const PoolView &P, const RowBatch &rows, const TokenIO &io, int d,
                               float *temp, cudaStream_t s) {
  if (d == 128) return run_tempstate<KT, VARIANT, 128>(P, rows, io, temp, s);
  if (d == 64) return run_tempstate<KT, VARIANT, 64>(P, rows, io, temp, s);
  return kUnsupported;
}

template <typename KT>
static cudaError_t tempstate_variant(const PoolView &P, const RowBatch &rows, const TokenIO &io,
                                     int variant, int d, float *temp, cudaStream_t s) {
  switch (variant) {
    case kPlain: return tempstate_d<KT, kPlain>(P, rows, io, d, temp, s);
    case kGated: return tempstate_d<KT, kGated>(P, rows, io, d, temp, s);
    case kGatedDelta: return tempstate_d<KT, kGatedDelta>(P, rows, io, d, temp, s);
  }
  return kUnsupported;
}

cudaError_t launch_verify_tempstate(const PoolView &P, const RowBatch &rows, const TokenIO &io,
                                    int variant, int dtype, int d, float *temp,
                                    cudaStream_t stream) {
  if (rows.count <= 0) return cudaSuccess;
  if (dtype == 0) return tempstate_variant<float>(P, rows, io, variant, d, temp, stream);
  if (dtype == 1) return tempstate_variant<__nv_bfloat16>(P, rows, io, variant, d, temp, stream);
  return kUnsupported;
}

cudaError_t launch_accept_tempstate(const PoolView &P, const RowBatch &rows, const float *temp,
                                    int T, int d, cudaStream_t stream) {
  if (rows.count <= 0) return cudaSuccess;
  dim3 grid(P.Hv, rows.count);
  tempstate_accept_kernel<<<grid, 256, 0, stream>>>(P, rows, temp, T, d, d);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ no allocation
// Temporary states for kvb_verify_tempstate_static: a fixed array inside the
// library, for callers that cannot allocate device memory.  Every GPU that
// loads the library holds it until the process exits.
constexpr size_t kStaticTempFloats = (size_t)KVB_STATIC_TEMP_BYTES / sizeof(float);
static __device__ __align__(256) float g_static_temp[kStaticTempFloats];

// Device address of g_static_temp on the current device.  Host code cannot use
// the array's name as a device address, so it is looked up once per device
// (with that device current) and cached.
static cudaError_t static_temp_address(float **out) {
  constexpr int kMaxDevices = 64;
  static std::mutex mu;
  static float *addr[kMaxDevices] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_static_temp);
    if (e != cudaSuccess) return e;
    addr[dev] = static_cast<float *>(p);
  }
  *out = addr[dev];
  return cudaSuccess;
}

cudaError_t launch_verify_tempstate_static(const PoolView &P, const RowBatch &rows,
                                           const TokenIO &io, int variant, int dtype, int d,
                                           cudaStream_t stream) {
  float *temp = nullptr;
  cudaError_t e = static_temp_address(&temp);
  if (e != cudaSuccess) return e;
  return launch_verify_tempstate(P, rows, io, variant, dtype, d, temp, stream);
}

cudaError_t launch_accept_tempstate_static(const PoolView &P, const RowBatch &rows, int T, int d,
                                           cudaStream_t stream) {
  float *temp = nullptr;
  cudaError_t e = static_temp_address(&temp);
  if (e != cudaSuccess) return e;
  return launch_accept_tempstate(P, rows, temp, T, d, stream);
}

}  // namespace kvb
