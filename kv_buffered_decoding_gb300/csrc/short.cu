// Short-context decode: outputs computed from the buffered keys and values
// alone, with no state (KVBuffer, "KVBuffer: IO-aware Serving for Linear
// Attention", abstract and "If this is right" section: short-context requests
// skip state creation and update entirely).  With S = 0 the decode formula
// reduces to attention over the buffer with decay weights:
//   u_t = v_t                                                 plain / gated
//   u_t = beta_t (v_t - sum_{i<t} e^{A_t-A_i} (k_t.k_i) u_i)   gated delta rule
//   o_t = sum_{i<t} e^{A_t-A_i} (q_t.k_i) u_i + (q_t.k_t) u_t
// One CTA of four warps per (batch row, value head).  Warp w takes buffered
// tokens w, w+4, w+8, ... in register chunks, issuing the next chunk's loads
// before computing the current one, reduces each chunk's dot products with one
// butterfly, and accumulates e^{A_t-A_i} s_i u_i for its lane's columns; the
// four warps' partial sums are added once through shared memory.
#include "kvb_device.cuh"

namespace kvb {

template <typename KT, int VARIANT, int D>
__global__ void __launch_bounds__(128) short_kernel(const PoolView P, const RowBatch rows,
                                                     const TokenIO io) {
  constexpr int NT = 128, NW = 4, E = D / 32;
  constexpr bool DELTA = VARIANT == kGatedDelta, GATED = VARIANT != kPlain;
  constexpr int C = DELTA ? 2 : 4;  // tokens per chunk (one butterfly of four sums)
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int h = blockIdx.x;
  const RowDesc d = rows.r[blockIdx.y];
  const size_t b = (size_t)rows.row0 + blockIdx.y;
  const int group = P.Hv / P.Hk;
  const int hq = h / group;
  const int n = d.n;  // buffered tokens; the current token goes to slot n

  __shared__ __align__(16) float qs[D];
  __shared__ __align__(16) float kts[D];
  __shared__ __align__(16) float part_o[NW][D];
  __shared__ __align__(16) float part_c[NW][D];
  __shared__ size_t koff[kMaxTok], voff[kMaxTok];
  __shared__ float s_t_s;
  __shared__ int bad;

  // 1. where tokens 0..n live; q (scaled) and k_t to shared
  if (warp == 0) {
    int anybad = 0;
    for (int i = lane; i <= n; i += 32) {
      const int g = buffer_row(P, d, i);
      anybad |= (g < 0);
      if (g >= 0) {
        koff[i] = kv_row(P, g, hq, P.Hk) * D;
        voff[i] = kv_row(P, g, h, P.Hv);
      }
    }
    anybad = __any_sync(kFull, anybad);
    if (lane == 0) bad = anybad;
  }
  const KT *qg = static_cast<const KT *>(io.q) + (b * P.Hk + hq) * D;
  const KT *kg = static_cast<const KT *>(io.k) + (b * P.Hk + hq) * D;
  for (int i = tid; i < D; i += NT) {
    qs[i] = P.scale * to_float(qg[i]);
    kts[i] = to_float(kg[i]);
  }
  float a_t = 0.f, beta_t = 0.f;
  if (GATED && io.log_g) a_t = io.log_g[b * P.Hv + h];
  if (DELTA) beta_t = io.beta[b * P.Hv + h];
  __syncthreads();
  if (bad) return;  // CTA-uniform

  const float A_t = (GATED && n > 0 ? P.gbuf[voff[n - 1]] : 0.f) + a_t;
  float qv[E], tv[E];
  load_smem<E>(qs + lane * E, qv);
  load_smem<E>(kts + lane * E, tv);
  if (warp == 0) {
    float st = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) st = fmaf(qv[e], tv[e], st);
    st = warp_sum(st);
    if (lane == 0) s_t_s = st;
  }

  // 2. this warp's buffered tokens, chunk by chunk with the next chunk in flight
  float po[E], pc[E];
#pragma unroll
  for (int e = 0; e < E; ++e) po[e] = pc[e] = 0.f;
  float kc[C][E], uc[C][E], ac[C];
  auto load_chunk = [&](int i0, float (&kk)[C][E], float (&uu)[C][E], float (&aa)[C]) {
#pragma unroll
    for (int x = 0; x < C; ++x) {
      const int i = i0 + NW * x;
      if (i < n) {
        load_row<E>(static_cast<const KT *>(P.kbuf) + koff[i] + lane * E, kk[x]);
        if (DELTA)
          load_row<E>(P.ubuf + voff[i] * D + lane * E, uu[x]);
        else
          load_row<E>(static_cast<const KT *>(P.vbuf) + voff[i] * D + lane * E, uu[x]);
        aa[x] = GATED ? P.gbuf[voff[i]] : 0.f;
      } else {
#pragma unroll
        for (int e = 0; e < E; ++e) kk[x][e] = uu[x][e] = 0.f;
        aa[x] = A_t;
      }
    }
  };
  const int stride = NW * C;  // tokens between this warp's chunks
  if (warp < n) load_chunk(warp, kc, uc, ac);
  for (int i0 = warp; i0 < n; i0 += stride) {
    float kn[C][E], un[C][E], an[C];
    const bool more = i0 + stride < n;
    if (more) load_chunk(i0 + stride, kn, un, an);
    float sums[4];
#pragma unroll
    for (int x = 0; x < C; ++x) {
      float sq = 0.f, sk = 0.f;
#pragma unroll
      for (int e = 0; e < E; ++e) {
        sq = fmaf(qv[e], kc[x][e], sq);
        if (DELTA) sk = fmaf(tv[e], kc[x][e], sk);
      }
      if (DELTA) {
        sums[2 * x] = sq;
        sums[2 * x + 1] = sk;
      } else {
        sums[x] = sq;
      }
    }
    const float r = butterfly4(sums[0], sums[1], sums[2], sums[3], lane);
    const float tot[4] = {__shfl_sync(kFull, r, 0), __shfl_sync(kFull, r, 8),
                          __shfl_sync(kFull, r, 16), __shfl_sync(kFull, r, 24)};
#pragma unroll
    for (int x = 0; x < C; ++x) {
      const float w = GATED ? expf(A_t - ac[x]) : 1.f;
      const float ws = w * (DELTA ? tot[2 * x] : tot[x]);
      const float wc = DELTA ? w * tot[2 * x + 1] : 0.f;
#pragma unroll
      for (int e = 0; e < E; ++e) {
        po[e] = fmaf(ws, uc[x][e], po[e]);
        if (DELTA) pc[e] = fmaf(wc, uc[x][e], pc[e]);
      }
    }
    if (more) {
#pragma unroll
      for (int x = 0; x < C; ++x) {
        ac[x] = an[x];
#pragma unroll
        for (int e = 0; e < E; ++e) {
          kc[x][e] = kn[x][e];
          uc[x][e] = un[x][e];
        }
      }
    }
  }
#pragma unroll
  for (int e = 0; e < E; ++e) {
    part_o[warp][lane * E + e] = po[e];
    part_c[warp][lane * E + e] = pc[e];
  }
  __syncthreads();

  // 3. one thread per column: the current token's u and the output; append
  const KT *vg = static_cast<const KT *>(io.v) + (b * P.Hv + h) * D;
  for (int c = tid; c < D; c += NT) {
    float o = 0.f, pcs = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      o += part_o[w][c];
      if (DELTA) pcs += part_c[w][c];
    }
    const float vt = to_float(vg[c]);
    float ut = vt;
    if (DELTA) ut = beta_t * (vt - pcs);
    o = fmaf(s_t_s, ut, o);
    io.o[(b * P.Hv + h) * D + c] = o;
    static_cast<KT *>(P.vbuf)[voff[n] * D + c] = static_cast<KT>(vt);
    if (DELTA) P.ubuf[voff[n] * D + c] = ut;
  }
  if (h % group == 0)
    for (int c = tid; c < D / 4; c += NT)
      st4(static_cast<KT *>(P.kbuf) + koff[n] + 4 * c, *reinterpret_cast<const float4 *>(&kts[4 * c]));
  if (tid == 0) {
    P.gbuf[voff[n]] = GATED ? A_t : 0.f;  // cumulative
    P.bbuf[voff[n]] = beta_t;
    if (h == 0) P.dlen[d.req] = n + 1;
  }
}

template <typename KT, int VARIANT>
static cudaError_t short_d(const PoolView &P, const RowBatch &rows, const TokenIO &io, int d,
                           cudaStream_t s) {
  dim3 grid(P.Hv, rows.count);
  if (d == 128) short_kernel<KT, VARIANT, 128><<<grid, 128, 0, s>>>(P, rows, io);
  else if (d == 64) short_kernel<KT, VARIANT, 64><<<grid, 128, 0, s>>>(P, rows, io);
  else return kUnsupported;
  return cudaGetLastError();
}

template <typename KT>
static cudaError_t short_variant(const PoolView &P, const RowBatch &rows, const TokenIO &io,
                                 int variant, int d, cudaStream_t s) {
  switch (variant) {
    case kPlain: return short_d<KT, kPlain>(P, rows, io, d, s);
    case kGated: return short_d<KT, kGated>(P, rows, io, d, s);
    case kGatedDelta: return short_d<KT, kGatedDelta>(P, rows, io, d, s);
  }
  return kUnsupported;
}

cudaError_t launch_short(const PoolView &P, const RowBatch &rows, const TokenIO &io, int variant,
                         int dtype, int d, cudaStream_t stream) {
  if (rows.count <= 0) return cudaSuccess;
  if (dtype == 0) return short_variant<float>(P, rows, io, variant, d, stream);
  if (dtype == 1) return short_variant<__nv_bfloat16>(P, rows, io, variant, d, stream);
  return kUnsupported;
}

}  // namespace kvb
