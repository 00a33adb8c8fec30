// Deferred state update: fold every buffered token of a request into its state.
//
// KVBuffer ("KVBuffer: IO-aware Serving for Linear Attention", Figure 1
// caption): when the buffer is full, the state is updated with all buffered
// KVs on the GPU and written back to the state slot.  For L buffered tokens
// with cumulative log-gates A_1..A_L (stored in the buffer) and pseudo-values u_i (u_i = v_i except
// for the gated delta rule, where u_i was computed when the token entered the
// buffer):
//     S <- e^{A_L} S0 + sum_{i<=L} e^{A_L-A_i} k_i u_i^T
// a rank-L update, K^T diag(w) U, of the register-resident state tile (two
// CTAs per head at d = 128, 16 consecutive rows per lane as in decode).  At
// L <= 64 this is 2 L flop per state element against 8 bytes of state traffic
// per element (read + write), i.e. below the fp32 FMA ridge: the kernel is
// bound by HBM.  Above rank 4 the update runs as mma.sync tf32 products on the
// register tile in place (fold_tile, kvb_device.cuh), which issues far fewer
// instructions than the FMAs.
//
// Used by kvb_flush, by kvb_accept when accepted drafts fill the buffer and by
// kvb_promote (rows flagged kFlagFromZero start from S = 0); decode folds
// in-kernel (decode.cu).
#include <type_traits>

#include "kvb_device.cuh"

namespace kvb {

template <typename KT, int VARIANT, int D, int NSPLIT>
__global__ void __launch_bounds__(2 * D / NSPLIT, 512 / (2 * D / NSPLIT))
    flush_kernel(const PoolView P, const RowBatch rows) {
  constexpr int DK = D, DV = D, NT = 2 * D / NSPLIT, RPT = DK / 8;
  constexpr int CW = DV / NSPLIT;
  constexpr bool DELTA = VARIANT == kGatedDelta;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int h = blockIdx.x / NSPLIT, part = blockIdx.x % NSPLIT;
  const int rsub = lane >> 2, row0 = rsub * RPT;
  const int colL = warp * 16 + (lane & 3) * 4, col0 = part * CW + colL;
  const RowDesc d = rows.r[blockIdx.y];
  const int hq = h / (P.Hv / P.Hk);
  const int L = d.n;

  // staged rows in the orders of fold_tile (kvb_device.cuh)
  constexpr int KST = DK + 8, UST = CW + 8;
  extern __shared__ float4 dyn_smem[];
  float *ks = reinterpret_cast<float *>(dyn_smem);  // [L][KST] keys
  float *us = ks + (size_t)L * KST;                 // [L][UST] u_i for this CTA's columns
  __shared__ float wt[kMaxTok];
  __shared__ size_t koff[kMaxTok], voff[kMaxTok];
  __shared__ float eL_s;
  __shared__ int bad;

  float *Sp = P.state + ((size_t)d.slot * P.Hv + h) * DK * DV;
  float4 s[RPT];
  if (d.flags & kFlagFromZero) {  // promotion: the slot's contents are not a state yet
#pragma unroll
    for (int j = 0; j < RPT; ++j) s[j] = f4(0.f);
  } else {
#pragma unroll
    for (int j = 0; j < RPT; ++j) s[j] = ld_stream4(Sp + (row0 + j) * DV + col0);
  }

  if (warp == 0) {
    int anybad = 0;
    for (int i = lane; i < L; i += 32) {
      const int g = buffer_row(P, d, i);
      anybad |= (g < 0);
      if (g >= 0) {
        koff[i] = kv_row(P, g, hq, P.Hk) * DK;
        voff[i] = kv_row(P, g, h, P.Hv);
      }
    }
    anybad = __any_sync(kFull, anybad);
    if (lane == 0) bad = anybad;
  }
  __syncthreads();
  if (bad) return;

  // weights from the stored cumulative log-gates (warp 0); keys to shared (all)
  if (warp == 0) {
    if (VARIANT != kPlain) {
      const float AL = P.gbuf[voff[L - 1]];
      for (int i = lane; i < L; i += 32) wt[i] = expf(AL - P.gbuf[voff[i]]);
      if (lane == 0) eL_s = expf(AL);
    } else {
      for (int i = lane; i < L; i += 32) wt[i] = 1.f;
      if (lane == 0) eL_s = 1.f;
    }
  }
  for (int idx = tid; idx < L * (DK / 4); idx += NT) {
    const int i = idx / (DK / 4), c = (idx % (DK / 4)) * 4;  // rows c .. c + 3
    const float4 k4 = ld4(static_cast<const KT *>(P.kbuf) + koff[i] + c);
    *reinterpret_cast<float2 *>(&ks[(size_t)i * KST + fold_kpos<RPT>(c)]) = make_float2(k4.x, k4.y);
    *reinterpret_cast<float2 *>(&ks[(size_t)i * KST + fold_kpos<RPT>(c + 2)]) = make_float2(k4.z, k4.w);
  }
  for (int idx = tid; idx < L * (CW / 4); idx += NT) {
    const int i = idx / (CW / 4), c = (idx % (CW / 4)) * 4;
    float4 u;
    if (DELTA)
      u = ld4(P.ubuf + voff[i] * DV + part * CW + c);
    else
      u = ld4(static_cast<const KT *>(P.vbuf) + voff[i] * DV + part * CW + c);
    fold_stage_u(&us[(size_t)i * UST + c], u);
  }
  __syncthreads();  // weights, keys and values staged

  // S <- e^{A_L} S0 + sum_i k_i (w_i u_i)^T
  const float eL = eL_s;
#pragma unroll
  for (int j = 0; j < RPT; ++j) s[j] = mul4(eL, s[j]);
  fold_tile<RPT, std::is_same<KT, __nv_bfloat16>::value>(s, ks, KST, us, UST, warp * 16, wt, L - 1,
                                                          lane);
#pragma unroll
  for (int j = 0; j < RPT; ++j) st_stream4(Sp + (row0 + j) * DV + col0, s[j]);
  if (h == 0 && part == 0 && tid == 0) P.dlen[d.req] = 0;
}

template <typename KT, int VARIANT, int D>
static cudaError_t run_flush(const PoolView &P, const RowBatch &rows, int max_len,
                             cudaStream_t stream) {
  constexpr int NS = D == 128 ? 2 : 1;
  const size_t smem = (size_t)max_len * ((D + 8) + (D / NS + 8)) * sizeof(float);
  cudaError_t e = ensure_smem((const void *)flush_kernel<KT, VARIANT, D, NS>, smem);
  if (e != cudaSuccess) return e;
  dim3 grid(P.Hv * NS, rows.count);
  flush_kernel<KT, VARIANT, D, NS><<<grid, 2 * D / NS, smem, stream>>>(P, rows);
  return cudaGetLastError();
}

template <typename KT, int VARIANT>
static cudaError_t flush_d(const PoolView &P, const RowBatch &rows, int d, int max_len,
                           cudaStream_t s) {
  if (d == 128) return run_flush<KT, VARIANT, 128>(P, rows, max_len, s);
  if (d == 64) return run_flush<KT, VARIANT, 64>(P, rows, max_len, s);
  return kUnsupported;
}

template <typename KT>
static cudaError_t flush_variant(const PoolView &P, const RowBatch &rows, int variant, int d,
                                 int max_len, cudaStream_t s) {
  switch (variant) {
    case kPlain: return flush_d<KT, kPlain>(P, rows, d, max_len, s);
    case kGated: return flush_d<KT, kGated>(P, rows, d, max_len, s);
    case kGatedDelta: return flush_d<KT, kGatedDelta>(P, rows, d, max_len, s);
  }
  return kUnsupported;
}

cudaError_t launch_flush(const PoolView &P, const RowBatch &rows, int variant, int dtype, int d,
                         int max_len, cudaStream_t stream) {
  if (rows.count <= 0) return cudaSuccess;
  if (d == 128 && max_len <= kStageTok && flush_stream_pays(rows.count * P.Hv, variant, dtype))
    return launch_flush_stream(P, rows, variant, dtype, stream);
  if (dtype == 0) return flush_variant<float>(P, rows, variant, d, max_len, stream);
  if (dtype == 1) return flush_variant<__nv_bfloat16>(P, rows, variant, d, max_len, stream);
  return kUnsupported;
}

}  // namespace kvb
